// msa_decode_step: the whole decode / verify step in one call -- plan, index
// scores, top-k selection, split-K sparse decode, combine -- as five kernels
// chained with programmatic dependent launch.
#include "msa_internal.cuh"

extern "C" msa_status msa_decode_step(const msa_config* cfg, void* ws, int32_t batch,
                                      const int32_t* seq_lens, const int32_t* block_table,
                                      int32_t bt_stride, const void* idx_q,
                                      const void* idx_k_pages, const void* q,
                                      const void* k_pages, const void* v_pages,
                                      float* block_scores, int32_t* selected, void* out,
                                      float* lse, msa_stream_t stream) {
  msa_status st = msa::check_config(cfg);
  if (st != MSA_OK) return st;
  if (msa::is_prefill(*cfg)) return MSA_ERR_INVALID_ARG;
  if (!ws || !idx_q || !idx_k_pages || !q || !k_pages || !v_pages || !block_scores ||
      !selected || !out || !lse)
    return MSA_ERR_INVALID_ARG;
  if ((st = msa_plan(cfg, batch, seq_lens, nullptr, block_table, bt_stride, ws, stream)) != MSA_OK)
    return st;
  if ((st = msa_index_score_topk(cfg, ws, idx_q, idx_k_pages, block_scores, selected,
                                 stream)) != MSA_OK)
    return st;
  if ((st = msa_sparse_decode(cfg, ws, q, k_pages, v_pages, selected, stream)) != MSA_OK)
    return st;
  return msa_combine(cfg, ws, out, lse, stream);
}
