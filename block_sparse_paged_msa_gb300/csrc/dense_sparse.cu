// msa_compact_selected: the compaction step of the dense-sparse decode.
//
// sglang minimax_sparse_backend.py (MiniMaxSparseAttnBackend.forward_decode,
// the use_dense_sparse_decode branch, and _dense_sparse_main_decode) turns the
// selected blocks into a page table and a real sequence length per query and
// runs a dense paged decode over it (trtllm batch decode, max_seq_len =
// topk_blocks * block_size).  Here one list per (token, KV head): the pages of
// its selected blocks in ascending block order (the plan's validated block
// table; blocks whose page the plan flagged are left out) and the number of
// keys they hold for the token -- every selected block is full except the
// token's own, which comes last -- so that msa_paged_decode, a dense paged
// decode over (page list, length), reads exactly the keys the sparse decode
// reads, in the same order.
//
// One warp per (token, KV head): the selected list S slots at a time, a
// ballot compacts the usable slots, a warp sum counts the keys.
#include "msa_internal.cuh"

namespace msa {
namespace {

__global__ void __launch_bounds__(256)
compact_kernel(WsView ws, int Hkv, int max_blocks, int S, const int32_t* __restrict__ selected,
               int32_t* __restrict__ page_table, int32_t* __restrict__ dense_len) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);   // (token, KV head)
  griddep_launch_dependents();
  griddep_wait();
  if (row >= (int64_t)ws.hdr->num_tokens * Hkv) return;               // warp-uniform
  const int t = (int)(row / Hkv);
  const int r = ws.tok_req[t];
  const int pos = r >= 0 ? ws.tok_pos[t] : -1;
  int32_t* out = page_table + row * S;
  int n = 0, cnt = 0;
  for (int base = 0; base < S; base += 32) {
    const int i = base + lane;
    int page = -1, vis = 0;
    if (r >= 0 && i < S) {
      const int j = selected[row * S + i];
      if (j >= 0 && j * kBlock <= pos) {
        page = ws.block_table[(int64_t)r * max_blocks + j];
        vis = min(kBlock, pos + 1 - j * kBlock);
      }
    }
    const bool ok = page >= 0;
    const unsigned m = __ballot_sync(0xffffffffu, ok);
    if (ok) out[cnt + __popc(m & ((1u << lane) - 1u))] = page;
    cnt += __popc(m);
    n += ok ? vis : 0;
  }
  for (int i = cnt + lane; i < S; i += 32) out[i] = -1;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
  if (lane == 0) dense_len[row] = n;
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" msa_status msa_compact_selected(const msa_config* cfg, const void* ws,
                                           const int32_t* selected, int32_t* page_table,
                                           int32_t* seq_lens, msa_stream_t stream) {
  msa_status st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (is_prefill(*cfg)) return MSA_ERR_INVALID_ARG;
  if (!ws || !selected || !page_table || !seq_lens) return MSA_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)max_tokens_of(*cfg) * cfg->num_kv_heads;
  if (rows <= 0) return MSA_OK;
  const int64_t grid = (rows + 7) / 8;
  if (grid > 0x7fffffff) return MSA_ERR_UNSUPPORTED;
  return launch_pdl(compact_kernel, dim3((unsigned)grid), dim3(256), 0, (cudaStream_t)stream,
                    view_of(*cfg, ws), cfg->num_kv_heads, cfg->max_blocks_per_req,
                    width_of(*cfg), selected, page_table, seq_lens);
}
