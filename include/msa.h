/*
 * msa.h -- C ABI of libmsa: block-sparse attention over a paged KV cache
 * (MiniMax-M3 style "MSA"), hand-written CUDA for sm_103a (GB300).
 *
 * The method (sglang minimax_sparse_backend.py, MiniMaxSparseAttnBackend:
 * __init__, forward_decode, forward_extend; vLLM
 * minimax_m3/nvidia/sparse_attention_msa.py, MiniMaxM3SparseMSAImpl.forward):
 * every query token rates each 128-token KV block of its request with a
 * low-dimensional index query/key, keeps the init blocks, the local blocks and
 * the topk_blocks best remaining blocks, and attends over those blocks only
 * (GQA: the query heads of one KV head share its selection).  A decode step is
 *
 *     msa_plan -> msa_index_score -> msa_topk_select -> msa_sparse_decode -> msa_combine
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All pointers are DEVICE pointers unless a comment says "host".  The caller
 *    owns every buffer; the library never allocates or frees device memory and
 *    never synchronises, except msa_check_device_error.
 *  - Work is enqueued on the caller's stream (NULL = legacy default stream).
 *    Every launch has a grid fixed by the msa_config maxima, and no call reads
 *    device data on the host, so the whole step can be captured in a CUDA graph
 *    once and replayed with new data in the same buffers.
 *  - Layouts (row-major, contiguous):
 *      q            [T, H_q, D]            bf16
 *      idx_q        [T, H_kv, d]           bf16
 *      k_pages      [num_pages, H_kv, P, D] bf16, or fp8 e4m3 codes (kv_dtype),
 *                   or NVFP4 slots [num_pages, 2 H_kv, P, 72] (MSA_KV_NVFP4)
 *      v_pages      [num_pages, H_kv, P, D] same type as k_pages
 *      idx_k_pages  [num_pages, H_kv, P, d] bf16
 *      block_table  [batch, >= max_blocks_per_req] int32 (row stride given);
 *                   entry j = physical page of the request's logical block j
 *      block_scores [T, H_kv, max_blocks_per_req] float
 *      selected     [T, H_kv, S] int32, S = init + local + topk blocks,
 *                   ascending block indices, padded with -1
 *      out          [T, H_q, D] bf16;  lse [T, H_q] float (natural log)
 *    T is the number of query tokens of the step (batch * q_len for decode and
 *    verify, cu_seqlens_q[batch] for prefill); P = block_size = page size = 128.
 *  - seq_lens[r] counts request r's KV tokens INCLUDING its new query tokens
 *    (the fused KV / index-K cache write precedes attention in forward_decode);
 *    the i-th of the n new tokens of request r sits at position
 *    seq_lens[r] - n + i and sees the tokens at positions <= its own.
 *  - A request with seq_len 0 (or a batch of 0) produces out = 0, lse = -inf
 *    (the idle-batch convention of forward_decode).
 *  - Errors: argument problems found on the host return a status before any
 *    launch.  Problems only visible on the device (a page id outside
 *    [0, num_pages), a seq_len above max_blocks_per_req * P or below the
 *    request's query count) never fault: the kernels skip the bad entry, set a
 *    bit in the workspace's error word, and msa_check_device_error reports it.
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* msa_stream_t;

typedef enum msa_status {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad stride ...   */
  MSA_ERR_UNSUPPORTED = 2,   /* valid, but outside what the kernels implement */
  MSA_ERR_CUDA = 3,          /* a CUDA runtime call failed                    */
  MSA_ERR_DEVICE_FLAG = 4    /* a kernel flagged bad data (see error bits)    */
} msa_status;

typedef enum msa_kv_dtype {
  MSA_KV_BF16 = 0,
  MSA_KV_FP8_E4M3 = 1,       /* e4m3 "fn" codes; value = decode(code) * scale */
  MSA_KV_NVFP4 = 2           /* NVFP4 slots (vLLM MiniMaxM3SparseMSANvfp4Backend):
                                each pool is [num_pages, 2 * H_kv, P, 72] bytes,
                                slot 2h = keys, slot 2h + 1 = values of KV head
                                h; a 72-byte token row is 64 bytes of FP4 E2M1
                                codes (element 2i in the low nibble of byte i)
                                then 8 E4M3 scales, one per 16 elements; value
                                = e2m1(code) * e4m3(block scale) * k_scale or
                                v_scale.  Keys are read from k_pages, values
                                from v_pages (the same combined pool is passed
                                twice).  Decode / verify only.                */
} msa_kv_dtype;

typedef enum msa_mode {
  MSA_MODE_DECODE = 0,       /* q_len new tokens per request (1 = decode, 2..4 =
                                speculative verify); msa_sparse_decode          */
  MSA_MODE_PREFILL = 1       /* a chunk of any length per request, given by
                                cu_seqlens_q; msa_build_k2q_csr +
                                msa_sparse_prefill; H_q / H_kv must divide 16     */
} msa_mode;

/* Bits of the device error word (msa_check_device_error). */
enum {
  MSA_DEVERR_PAGE_RANGE = 1,   /* block table / req_to_token page outside the pool */
  MSA_DEVERR_SEQ_LEN = 2,      /* seq_len > max_blocks_per_req*P, or < query count,
                                  or the step's tokens exceed max_q_tokens        */
  MSA_DEVERR_SLOT_ALIGN = 4,   /* req_to_token slot of a block not page-aligned   */
  MSA_DEVERR_TIMEOUT = 8,      /* a pipeline wait gave up (results invalid)       */
  MSA_DEVERR_FP16_RANGE = 16   /* a bf16 value beyond the fp16 range (|x| > 65504,
                                  or infinite) met an fp16 operand: the queries
                                  of the fp8 / NVFP4 decode, the values of the
                                  prefill tiles (results involving it invalid).
                                  Magnitudes below 2^-14 are not flagged; they
                                  keep fp16's subnormal precision only.          */
};

/*
 * Static configuration of one sparse-attention layer and of the largest step
 * the workspace must hold.  Block counts follow sglang
 * MiniMaxSparseAttnBackend.__init__: init_blocks = ceil(sparse_init_tokens/P)
 * (or sparse_init_block), local_blocks = ceil(sparse_local_tokens/P) + 1 (or
 * sparse_local_block), topk_blocks = sparse_topk_blocks, index_dim =
 * sparse_index_dim.  GQA: num_q_heads / num_kv_heads query heads per KV head
 * (qhead_per_kv in MiniMaxM3SparseMSAImpl.forward).
 */
typedef struct msa_config {
  int32_t num_q_heads;        /* H_q                                            */
  int32_t num_kv_heads;       /* H_kv; H_q % H_kv == 0, H_q / H_kv <= 16         */
  int32_t head_dim;           /* D; must be 128                                  */
  int32_t block_size;         /* P = sparse block = KV page; must be 128         */
  int32_t init_blocks;        /* >= 0                                            */
  int32_t local_blocks;       /* >= 1 (includes the query's own block)           */
  int32_t topk_blocks;        /* >= 0                                            */
  int32_t index_dim;          /* d; 64 or 128                                    */
  int32_t q_len;              /* new query tokens per request: 1 = decode,
                                 2..4 = speculative verify                       */
  int32_t kv_dtype;           /* msa_kv_dtype                                    */
  float softmax_scale;        /* applied to q.k before the softmax               */
  float k_scale;              /* fp8 / nvfp4: dequantised k = code value * k_scale */
  float v_scale;              /* fp8 / nvfp4: dequantised v = code value * v_scale */
  int32_t max_batch;          /* largest batch a plan may describe               */
  int32_t max_q_tokens;       /* largest T; 0 = max_batch * q_len                */
  int32_t max_blocks_per_req; /* block-table width used; seq_len <= this * P     */
  int32_t num_pages;          /* pages in the KV / index-K pool                  */
  int32_t blocks_per_split;   /* selected blocks per split-K work item; 0 = auto */
  int32_t mode;               /* msa_mode: decode / verify, or chunked prefill   */
} msa_config;

/* Human-readable name of a status (static string). */
const char* msa_status_string(msa_status status);

/*
 * Block counts from token counts, as sglang MiniMaxSparseAttnBackend.__init__
 * resolves a layer's sparse configuration when it gives tokens instead of
 * blocks:
 *   msa_init_blocks_from_tokens(n, P)  = ceil(n / P)      (sparse_init_tokens)
 *   msa_local_blocks_from_tokens(n, P) = ceil(n / P) + 1  (sparse_local_tokens;
 *                                        the query's own, partly filled block
 *                                        comes on top of the window)
 * Host-only, no GPU needed.  Return -1 if n < 0 or P <= 0.
 */
int32_t msa_init_blocks_from_tokens(int32_t tokens, int32_t block_size);
int32_t msa_local_blocks_from_tokens(int32_t tokens, int32_t block_size);

/* MSA_OK if the kernels implement cfg, else INVALID_ARG / UNSUPPORTED.  Every
 * entry point below runs this check first. */
msa_status msa_validate_config(const msa_config* cfg);

/* Width S of a selected list: init_blocks + local_blocks + topk_blocks. */
int32_t msa_selected_width(const msa_config* cfg);

/* Number of split-K partials per (token, query head) msa_sparse_decode writes. */
int32_t msa_num_splits(const msa_config* cfg);

/* Bytes of device workspace a step needs (plan metadata, a validated copy of
 * the block table, split-K partials).  0 if cfg is not valid.  The workspace
 * must be 256-byte aligned; its contents need no initialisation. */
size_t msa_workspace_bytes(const msa_config* cfg);

/*
 * msa_plan -- split metadata for one step, built on the device
 * (sglang MiniMaxSparseAttnBackend._prepare_msa_decode_meta: the decode plan is
 * built per batch outside graph capture and refreshed in place; vLLM
 * MiniMaxM3SparseMSAMetadataBuilder.build: block_table + seq_lens +
 * decode_query_len).
 *   batch        host int, 0 <= batch <= cfg->max_batch
 *   seq_lens     [batch] int32
 *   cu_seqlens_q [batch + 1] int32 or NULL; NULL = cfg->q_len tokens per request
 *   block_table  [batch, bt_stride] int32; bt_stride >= cfg->max_blocks_per_req
 *   ws           workspace of msa_workspace_bytes(cfg) bytes
 * Writes per-request block counts and their prefix sums, per-token (request,
 * position), and a validated copy of the block table into ws; resets the
 * device error word.  Entries past a request's last block are not read.
 */
msa_status msa_plan(const msa_config* cfg, int32_t batch, const int32_t* seq_lens,
                    const int32_t* cu_seqlens_q, const int32_t* block_table,
                    int32_t bt_stride, void* ws, msa_stream_t stream);

/*
 * msa_plan_from_req_to_token -- as msa_plan, but the block table is derived
 * from sglang's token-slot map (MiniMaxSparseAttnBackend._prepare_msa_decode_meta
 * feeds req_to_token and req_pool_indices to update_msa_decode_cg_meta):
 * page of block j of request r = req_to_token[req_pool_indices[r], j * P] / P.
 *   req_to_token      [pool_rows, r2t_stride] int32 token slots
 *   req_pool_indices  [batch] int64 rows of req_to_token
 * A slot that is not a multiple of P sets MSA_DEVERR_SLOT_ALIGN.
 */
msa_status msa_plan_from_req_to_token(const msa_config* cfg, int32_t batch,
                                      const int32_t* seq_lens,
                                      const int32_t* cu_seqlens_q,
                                      const int32_t* req_to_token, int32_t r2t_stride,
                                      const int64_t* req_pool_indices, void* ws,
                                      msa_stream_t stream);

/*
 * msa_cache_write -- stores the step's new keys, values and index keys into
 * the paged pools before attention (sglang MiniMaxSparseAttnBackend
 * forward_decode / forward_extend call set_fused_kv_index_buffer(layer,
 * out_cache_loc, k, v, idx_k, idx_v) first; that is why seq_lens counts the
 * new tokens).  Run it after msa_plan and before msa_index_score of the same
 * step, on the same workspace.
 *   out_cache_loc  [T] int64 token slots, slot = page * P + row, or NULL: the
 *                  slot comes from the plan -- token i of request r (position
 *                  seq_len - n + i) goes to row pos % P of the page the block
 *                  table maps block pos / P to
 *   k, v           [T, H_kv, D] bf16;  idx_k [T, H_kv, d] bf16 or NULL (no
 *                  index-key write);  idx_v [T, H_kv, d] bf16 or NULL (no
 *                  index-value write: layers without the index-value branch)
 *   k_pages, v_pages, idx_k_pages: the pools (layouts above); idx_v_pages
 *                  [num_pages, H_kv, P, d] bf16, the index-value pool
 * bf16 pools store the values as they are.  e4m3 pools store, per value, the
 * e4m3fn code nearest to x / scale (cfg->k_scale or v_scale; one IEEE fp32
 * division), ties to even, magnitudes beyond 448 saturated to +-448, NaN kept.
 * NVFP4 pools (k_pages and v_pages may be the same allocation) take the keys
 * of KV head h in slot 2h of k_pages and the values in slot 2h + 1 of
 * v_pages.  The pages give the format, not the quantiser; this library's
 * reading: each 16-element block's scale byte is the e4m3fn code of
 * amax / (6 * scale), each element the E2M1 code of x / (e4m3(scale byte) *
 * scale), every division and product one IEEE fp32 operation and every code
 * round-to-nearest-even, saturating; a block whose scale code is 0 stores zero
 * codes.  E2M1 has no NaN: a NaN element is stored as +6 (its block's scale
 * comes from the other elements).
 * Tokens of idle requests are skipped.  A slot outside [0, num_pages * P) is
 * skipped and sets MSA_DEVERR_PAGE_RANGE.  All pointers 16-byte aligned.
 */
msa_status msa_cache_write(const msa_config* cfg, void* ws, const int64_t* out_cache_loc,
                           const void* k, const void* v, const void* idx_k, const void* idx_v,
                           void* k_pages, void* v_pages, void* idx_k_pages, void* idx_v_pages,
                           msa_stream_t stream);

/*
 * msa_index_attention -- the index-value branch's output (sglang
 * MiniMaxSparseAttnBackend: layers outside disable_value_layer_ids keep an
 * index-value cache, get_index_kv_buffer, and the sparse ops return (idx_o, o)
 * with idx_o of shape [tokens, num_idx_heads * idx_head_dim]).  The pages do
 * not give idx_o's formula; this library's reading (its parity is unpinned):
 * the index head is a dense causal attention head,
 *   idx_o[t, h] = sum_u softmax_u(idx_q[t,h] . idx_k[u,h] / sqrt(d)) idx_v[u,h]
 * over the request's tokens u at positions <= position(t).  Decode mode, after
 * msa_plan (and msa_cache_write) of the step.
 *   idx_v_pages  [num_pages, H_kv, P, d] bf16
 *   scratch      msa_index_attention_scratch_bytes(cfg) bytes, 256-byte aligned
 *                (split partials; no initialisation needed)
 *   idx_out      [T, H_kv, d] bf16;  idx_lse [T, H_kv] float (natural log) or NULL
 * Idle tokens get idx_out = 0, idx_lse = -inf.  Blocks whose page the plan
 * flagged are skipped.
 */
size_t msa_index_attention_scratch_bytes(const msa_config* cfg);
msa_status msa_index_attention(const msa_config* cfg, const void* ws, const void* idx_q,
                               const void* idx_k_pages, const void* idx_v_pages, void* scratch,
                               void* idx_out, float* idx_lse, msa_stream_t stream);

/*
 * msa_index_score -- block scores from the index query/key
 * (sglang MiniMaxSparseAttnBackend.__init__ reads the index head dim and
 * score_type; forward_decode passes idx_q and the index-K cache to the sparse
 * decode op).  For every token t, KV head h and visible block j:
 *     block_scores[t, h, j] = max over tokens u of block j with
 *                             position(u) <= position(t) of  idx_q[t,h,:] . idx_k[u,h,:]
 * accumulated in fp32 (exact for the integer-valued index vectors used in
 * tests).  Entries j >= the token's visible block count are not written,
 * except in decode mode with one new token per request, where every entry of
 * the step's tokens is first set to -inf (the scan's two half-block units meet
 * there by an atomic max).
 * Decode mode: bandwidth-bound, every visible index key read once per request
 * (q_len <= 4 queries share each load).  Prefill mode: tensor-core tiles of
 * 128 query tokens x two 128-key blocks (tcgen05, fp32 accumulators in tensor
 * memory), causal.  idx_q and idx_k_pages must be 16-byte aligned.
 */
msa_status msa_index_score(const msa_config* cfg, const void* ws, const void* idx_q,
                           const void* idx_k_pages, float* block_scores,
                           msa_stream_t stream);

/*
 * msa_index_score_topk -- msa_index_score then msa_topk_select on the same
 * stream (the second launch overlaps the first one's tail), in one call.
 * Arguments, results and errors as in those two calls.  (A scan that selects
 * each request's rows as it finishes them, counting scored blocks per
 * (request, KV head), measured slower on GB300 than the separate selection
 * kernel: the per-block release of the counts and the selection tail at the
 * end of the scan cost more than the launch they save.)
 */
msa_status msa_index_score_topk(const msa_config* cfg, void* ws, const void* idx_q,
                                const void* idx_k_pages, float* block_scores, int32_t* selected,
                                msa_stream_t stream);

/*
 * msa_topk_select -- per (token, KV head): blocks [0, init) U [nb - local, nb)
 * U the topk best of the remaining blocks, ranked by score descending and block
 * index ascending on ties; written ascending into selected[t, h, 0..S), the
 * rest -1.  nb = position / P + 1.  (vLLM MiniMaxM3SparseMSAImpl.forward reads
 * the per-token [H, MK] selected-block lists that this produces.)
 */
msa_status msa_topk_select(const msa_config* cfg, const void* ws,
                           const float* block_scores, int32_t* selected,
                           msa_stream_t stream);

/*
 * msa_sparse_decode -- split-K flash decoding over the selected blocks only
 * (vLLM sparse_attention_msa.py module docstring and
 * MiniMaxM3SparseMSAImpl.forward: split-K decode over the top-k blocks with
 * block_table, seq_lens and decode_query_len; fp8 and NVFP4 KV are dequantised
 * on load, the NVFP4 pages read directly in their packed form).
 * For each token t, KV head h and split s, every query head of h's group runs
 * an online softmax over the tokens of the split's selected blocks that are at
 * or before t's position, and the normalised partial output and its
 * log-sum-exp are written to the workspace.  msa_combine finishes the step.
 */
msa_status msa_sparse_decode(const msa_config* cfg, void* ws, const void* q,
                             const void* k_pages, const void* v_pages,
                             const int32_t* selected, msa_stream_t stream);

/*
 * Dense-sparse decode (sglang MiniMaxSparseAttnBackend.forward_decode with
 * use_dense_sparse_decode, _dense_sparse_main_decode: the selected blocks
 * become a page table and a real sequence length per query, and a dense paged
 * decode runs over them with max_seq_len = topk_blocks * block_size).  The
 * pages do it for one KV head; here the lists are per (token, KV head).
 *
 * msa_compact_selected -- after msa_topk_select (decode mode): for every token
 * t and KV head h, page_table[t, h, 0..S) = the pages of selected[t, h, :]'s
 * blocks in ascending block order (blocks whose page the plan flagged are left
 * out), -1 after them, and seq_lens[t, h] = the number of keys they hold for
 * the token (every block full but the token's own, which is last).
 *   page_table [T, H_kv, S] int32;  seq_lens [T, H_kv] int32
 *
 * msa_paged_decode -- a dense paged decode over such lists (from
 * msa_compact_selected or built by the caller): for each token t and KV head
 * h, every query head of h's group attends to the first seq_lens[t, h] keys of
 * the pages page_table[t, h, 0..), page i holding keys i*P .. i*P + P - 1.
 * Split-K partials go to ws as for msa_sparse_decode; msa_combine finishes.
 * A listed page outside [0, num_pages) within the length is skipped and sets
 * MSA_DEVERR_PAGE_RANGE.  Run after msa_plan (it takes the step's tokens from
 * the plan).  Keys beyond S * P are not read.  All KV dtypes.
 */
msa_status msa_compact_selected(const msa_config* cfg, const void* ws, const int32_t* selected,
                                int32_t* page_table, int32_t* seq_lens, msa_stream_t stream);
msa_status msa_paged_decode(const msa_config* cfg, void* ws, const void* q, const void* k_pages,
                            const void* v_pages, const int32_t* page_table,
                            const int32_t* seq_lens, msa_stream_t stream);

/*
 * msa_combine -- log-sum-exp merge of the split-K partials in ws
 * (FlashMLA decode in sglang flashmla_backend.py returns (o, lse) per split
 * plan): lse = ln sum_s exp(lse_s), out = sum_s exp(lse_s - lse) o_s, out
 * rounded to bf16.  All splits empty -> out = 0, lse = -inf.  Decode mode
 * merges the splits of msa_sparse_decode; prefill mode the selected slots of
 * msa_sparse_prefill (each token's first min(nb, S) slots).  out must be
 * 8-byte aligned (decode) or 16-byte aligned (prefill).
 */
msa_status msa_combine(const msa_config* cfg, const void* ws, void* out, float* lse,
                       msa_stream_t stream);

/*
 * Key-block -> query CSR for prefill (vLLM MiniMaxM3SparseMSAImpl.forward calls
 * build_k2q_csr on the [H, tokens, MK] selections with qhead_per_kv).  Rows
 * sit on the fixed grid row = (h * max_batch + r) * max_blocks_per_req + j
 * (KV head h, request r, key block j), so every size depends on cfg alone;
 * rows of absent requests / blocks are empty.
 *   msa_k2q_rows(cfg)      number of rows (row_ptr holds rows + 1 int32)
 *   msa_k2q_capacity(cfg)  an upper bound of the entries (q_indices length)
 * msa_build_k2q_csr (prefill mode only) fills row_ptr (prefix sums, row_ptr[0]
 * = 0) and q_indices: row (h, r, j) lists, ascending, the token indices t of
 * request r whose selected[t, h, :] contains j (j visible to t).
 * Deterministic.  It also records in ws, for every (token, KV head, slot of
 * the selected list), the CSR entry that holds it, which msa_sparse_prefill's
 * output layout and msa_combine use: run it on the selections of this step,
 * after msa_plan, before msa_sparse_prefill.
 */
int64_t msa_k2q_rows(const msa_config* cfg);
int64_t msa_k2q_capacity(const msa_config* cfg);
msa_status msa_build_k2q_csr(const msa_config* cfg, const void* ws, const int32_t* selected,
                             int32_t* row_ptr, int32_t* q_indices, msa_stream_t stream);

/*
 * msa_sparse_prefill -- block-sparse causal attention for a prefill chunk
 * (vLLM MiniMaxM3SparseMSAImpl.forward: sparse_atten_func with blk_kv = 128,
 * causal = True, page_table and the CSR).  One tile per CSR row: the row's
 * tokens x their GQA query heads against the block's 128 keys, causal inside
 * the block that holds the token.  Writes one normalised fp16 partial and its
 * LSE per (CSR entry, query head of the entry's KV group) into ws, row entry *
 * G + g, so that a tile's rows are contiguous; msa_combine merges each token's
 * slots into out / lse.  selected is not read (the CSR build recorded what it
 * needs).  q, k_pages and v_pages must be 16-byte aligned.  Prefill mode, bf16
 * or NVFP4 KV (fp8 -> MSA_ERR_UNSUPPORTED).  NVFP4 (vLLM
 * MiniMaxM3SparseMSANvfp4Backend, whose prefill runs sparse_atten_nvfp4_kv_func):
 * k_pages and v_pages are the slot pools as for decode; each row's key and
 * value slots are dequantised in shared memory (keys to bf16, values to fp16,
 * both exact), k_scale scales the scores and v_scale the output.
 */
msa_status msa_sparse_prefill(const msa_config* cfg, void* ws, const void* q,
                              const void* k_pages, const void* v_pages,
                              const int32_t* selected, const int32_t* row_ptr,
                              const int32_t* q_indices, msa_stream_t stream);

/*
 * msa_sparse_decode_noalloc -- msa_plan + msa_sparse_decode + msa_combine in
 * one call that allocates nothing and takes no workspace.  The method's pages
 * have no counterpart; it exists for callers that cannot allocate device
 * memory (a host framework whose allocator owns all device memory, a serving
 * loop that reserved nearly all HBM for its KV cache, a latency-critical path
 * that cannot afford cudaMalloc / cudaFree).  The caller passes its inputs
 * (seq_lens, block_table as for msa_plan with cu_seqlens_q = NULL; q, k_pages,
 * v_pages; `selected` as msa_topk_select writes it, e.g. from its own indexer)
 * and its outputs (out, lse, as msa_combine writes them).
 * Scratch: a fixed device array of MSA_NOALLOC_SCRATCH_BYTES inside the
 * library, held by every GPU that loads the library until the process exits.
 * Returns MSA_ERR_UNSUPPORTED, before any launch, when the step needs more
 * than that (msa_workspace_bytes(cfg) > MSA_NOALLOC_SCRATCH_BYTES).
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  The cached address belongs to the device's primary context: do
 * not keep using the library on a device after cudaDeviceReset of it.  All
 * calls share the one array: calls whose work overlaps on the GPU (other
 * streams, other threads) race and must be serialised by the caller.  Each
 * call rewrites every part of the scratch it reads, so earlier contents never
 * leak into a result.  Data problems found on the device (bad page ids, a
 * seq_len out of range, a pipeline wait that gave up) are recorded in the
 * array's error words as for a workspace; msa_noalloc_check_device_error
 * reads them.
 */
#define MSA_NOALLOC_SCRATCH_BYTES (16u << 20)
msa_status msa_sparse_decode_noalloc(const msa_config* cfg, int32_t batch,
                                     const int32_t* seq_lens, const int32_t* block_table,
                                     int32_t bt_stride, const void* q, const void* k_pages,
                                     const void* v_pages, const int32_t* selected, void* out,
                                     float* lse, msa_stream_t stream);

/*
 * msa_noalloc_check_device_error -- msa_check_device_error for the scratch
 * array of msa_sparse_decode_noalloc on the current device: synchronises
 * `stream`, writes the OR of the error bits of the last no-alloc call into
 * *flags (host) and returns MSA_ERR_DEVICE_FLAG if any is set.  Allocates
 * nothing; never call it inside stream capture.
 */
msa_status msa_noalloc_check_device_error(int32_t* flags, msa_stream_t stream);

/*
 * msa_decode_step -- one decode / verify step (decode mode): msa_plan (with
 * cu_seqlens_q = NULL), msa_index_score_topk (msa_index_score +
 * msa_topk_select), msa_sparse_decode, msa_combine.
 * Arguments as in those calls.  The kernels are chained with programmatic
 * dependent launch, so each one's launch overlaps the previous one's tail.
 */
msa_status msa_decode_step(const msa_config* cfg, void* ws, int32_t batch,
                           const int32_t* seq_lens, const int32_t* block_table,
                           int32_t bt_stride, const void* idx_q, const void* idx_k_pages,
                           const void* q, const void* k_pages, const void* v_pages,
                           float* block_scores, int32_t* selected, void* out, float* lse,
                           msa_stream_t stream);

/*
 * msa_check_device_error -- synchronises `stream`, reads the workspace error
 * words (the plan's per-request words and the later kernels' word) into
 * *flags (host, OR of all) and returns MSA_ERR_DEVICE_FLAG if any bit is set.
 * Never call it inside stream capture.
 */
msa_status msa_check_device_error(const void* ws, int32_t* flags, msa_stream_t stream);

/*
 * msa_selftest_wait_timeout -- checks the failure path of the pipeline waits.
 * Launches one CTA that waits on an mbarrier nothing ever completes, through
 * the same bounded wait every warp-specialised kernel uses, with a short limit
 * (2^14 polls).  The wait gives up and sets MSA_DEVERR_TIMEOUT in the
 * workspace's error word, which msa_check_device_error then reports; no
 * device fault, and the context stays usable (msa_plan clears the word).
 * ws: a workspace of msa_workspace_bytes(cfg) bytes.  Asynchronous on `stream`.
 */
msa_status msa_selftest_wait_timeout(const msa_config* cfg, void* ws, msa_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MSA_H_ */
