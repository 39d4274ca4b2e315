// Internal definitions shared by the libmsa translation units: workspace layout,
// argument checks and small device helpers.  Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "../../include/msa.h"

namespace msa {

constexpr int kBlock = 128;      // P: sparse block = KV page
constexpr int kHeadDim = 128;    // D
constexpr int kFp4Row = kHeadDim / 2 + kHeadDim / 16;   // NVFP4 row: 64 code + 8 scale bytes
constexpr int kMaxGroup = 16;    // query heads per KV head (one m16 MMA tile)
constexpr int kMaxBlocksPerReq = 8192;
constexpr int kMaxBatch = 65536;

// Workspace header (first 256 bytes).
struct WsHeader {
  int32_t err;            // MSA_DEVERR_* bits of the kernels after the plan
  int32_t batch;
  int32_t num_tokens;     // T of the current plan
  int32_t total_blocks;   // sum over requests of ceil(seq_len / P)
  int32_t max_batch;      // number of plan_err words
  int32_t work_next;      // msa_sparse_decode: next work item to hand out
  int32_t work_done;      //   and CTAs done taking items (both zeroed by the plan
                          //   and by the last CTA of each launch)
};

inline size_t align_up(size_t x, size_t a = 256) { return (x + a - 1) / a * a; }

inline int32_t width_of(const msa_config& c) {
  return c.init_blocks + c.local_blocks + c.topk_blocks;
}

inline int32_t max_tokens_of(const msa_config& c) {
  return c.max_q_tokens > 0 ? c.max_q_tokens : c.max_batch * c.q_len;
}

int32_t blocks_per_split_of(const msa_config& c);  // resolves the 0 = auto case

inline bool is_prefill(const msa_config& c) { return c.mode == MSA_MODE_PREFILL; }

// Partials per (token, query head): split-K splits in decode mode, one per
// selected slot in prefill mode.
inline int32_t splits_of(const msa_config& c) {
  int32_t S = width_of(c);
  if (is_prefill(c)) return S > 0 ? S : 1;
  int32_t b = blocks_per_split_of(c);
  return S <= 0 ? 1 : (S + b - 1) / b;
}

// Bytes of one partial-output element: fp32 (decode), fp16 (prefill, where
// the per-slot partials dominate the traffic).
inline size_t part_elem_bytes(const msa_config& c) { return is_prefill(c) ? 2 : 4; }

// CSR rows of the key-block -> query map: (KV head, request, block) grid.
inline int64_t csr_rows_of(const msa_config& c) {
  return (int64_t)c.num_kv_heads * c.max_batch * c.max_blocks_per_req;
}

// Prefill CSR build: per (KV head, key block) a bitmap over the step's query
// tokens, request r's tokens from word (first token / 32) + r, so requests
// never share a word.  Words per (head, block):
inline int64_t csr_words_per_row(const msa_config& c) {
  return (int64_t)(max_tokens_of(c) + 31) / 32 + c.max_batch;
}
inline int64_t csr_words_of(const msa_config& c) {
  return (int64_t)c.num_kv_heads * c.max_blocks_per_req * csr_words_per_row(c);
}

// Upper bound of the sparse-prefill work items: one per CSR row plus one per
// 128 entries (an item holds at least 16 tiles of 8 tokens, unless it ends a row).
inline int64_t prefill_items_bound(const msa_config& c) {
  return csr_rows_of(c) + ((int64_t)max_tokens_of(c) * c.num_kv_heads * width_of(c) + 127) / 128 +
         1;
}

// Byte offsets of every workspace region.
struct WsLayout {
  size_t plan_err, req_seq_len, req_nb, req_cu_nb, req_qstart, tok_req, tok_pos, block_table;
  size_t sched, item_order, slot_entry, csr_bits, csr_wpre, o_part, lse_part, total;
};

inline WsLayout layout_of(const msa_config& c) {
  WsLayout L;
  const size_t B = (size_t)c.max_batch, T = (size_t)max_tokens_of(c);
  const size_t NS = (size_t)splits_of(c), Hq = (size_t)c.num_q_heads;
  size_t o = 256;
  L.plan_err = o;    o = align_up(o + 4 * (B > 0 ? B : 1));
  L.req_seq_len = o; o = align_up(o + 4 * B);
  L.req_nb = o;      o = align_up(o + 4 * B);
  L.req_cu_nb = o;   o = align_up(o + 4 * (B + 1));
  L.req_qstart = o;  o = align_up(o + 4 * (B + 1));
  L.tok_req = o;     o = align_up(o + 4 * T);
  L.tok_pos = o;     o = align_up(o + 4 * T);
  L.block_table = o; o = align_up(o + 4 * B * (size_t)c.max_blocks_per_req);
  L.sched = o;       o = align_up(o + (is_prefill(c) ? 4 * (size_t)(csr_rows_of(c) + 1) : 0));
  L.item_order = o;  o = align_up(o + (is_prefill(c) ? 16 * (size_t)prefill_items_bound(c) : 0));
  L.slot_entry = o;  o = align_up(o + (is_prefill(c) ? 4 * T * (size_t)c.num_kv_heads * width_of(c) : 0));
  L.csr_bits = o;    o = align_up(o + (is_prefill(c) ? 4 * csr_words_of(c) : 0));
  L.csr_wpre = o;    o = align_up(o + (is_prefill(c) ? 4 * csr_words_of(c) : 0));
  L.o_part = o;      o = align_up(o + part_elem_bytes(c) * T * Hq * NS * kHeadDim);
  L.lse_part = o;    o = align_up(o + 4 * T * Hq * NS);
  L.total = o;
  return L;
}

// Typed views of a workspace, passed to kernels by value.
struct WsView {
  WsHeader* hdr;
  int32_t* plan_err;      // [max_batch] error bits of each plan CTA, rewritten every plan
  int32_t* req_seq_len;
  int32_t* req_nb;
  int32_t* req_cu_nb;
  int32_t* req_qstart;
  int32_t* tok_req;
  int32_t* tok_pos;
  int32_t* block_table;   // [max_batch, max_blocks_per_req], -1 = invalid
  int32_t* sched;         // prefill: [csr rows + 1] first work item of each CSR row
  int4* item_order;       // prefill: work items by size, largest first: (CSR row,
                          // first entry, end entry, 0)
  int32_t* slot_entry;    // prefill: [T, H_kv, S] the CSR entry that holds (token, KV
                          // head, slot of the selected list)
  uint32_t* csr_bits;     // prefill: [H_kv, NB, words] token bitmaps of the CSR rows
  int32_t* csr_wpre;      // prefill: same shape, set bits before each word within its row
  // Partial outputs and their LSE.  Decode: [T, H_q, NS, D] fp32 and [T, H_q, NS]
  // (NS splits).  Prefill: fp16 rows indexed entry * G + g, where entry is the
  // CSR entry of (token, KV head h, block) and g the query head within h's
  // group, so an M-tile's rows are contiguous; [T * H_q * S] rows of D.
  void* o_part;
  float* lse_part;
};

inline WsView view_of(const msa_config& c, const void* ws) {
  WsLayout L = layout_of(c);
  char* b = (char*)ws;
  WsView v;
  v.hdr = (WsHeader*)b;
  v.plan_err = (int32_t*)(b + L.plan_err);
  v.req_seq_len = (int32_t*)(b + L.req_seq_len);
  v.req_nb = (int32_t*)(b + L.req_nb);
  v.req_cu_nb = (int32_t*)(b + L.req_cu_nb);
  v.req_qstart = (int32_t*)(b + L.req_qstart);
  v.tok_req = (int32_t*)(b + L.tok_req);
  v.tok_pos = (int32_t*)(b + L.tok_pos);
  v.block_table = (int32_t*)(b + L.block_table);
  v.sched = (int32_t*)(b + L.sched);
  v.item_order = (int4*)(b + L.item_order);
  v.slot_entry = (int32_t*)(b + L.slot_entry);
  v.csr_bits = (uint32_t*)(b + L.csr_bits);
  v.csr_wpre = (int32_t*)(b + L.csr_wpre);
  v.o_part = (void*)(b + L.o_part);
  v.lse_part = (float*)(b + L.lse_part);
  return v;
}

msa_status check_config(const msa_config* c);
// Tensor map of a row-major [rows, 128 columns] array (a KV pool viewed as
// num_pages * H_kv * 128 rows, or the queries as tokens * H_q rows): bf16 ->
// boxes of 64 columns x box_rows, e4m3 -> 128 x box_rows, 128-byte swizzle.
bool make_pool_map(CUtensorMap* m, const void* base, int64_t rows, bool fp8,
                   int box_rows = kBlock);
// General bf16 tensor map with 128-byte swizzle: dims / box innermost first,
// strides_bytes[i] = byte stride of dimension i + 1.
bool make_bf16_map(CUtensorMap* m, const void* base, int rank, const int64_t* dims,
                   const int64_t* strides_bytes, const int* box);
// Index scores of a prefill chunk (tensor-core tiles; prefill.cu).
msa_status prefill_index_score(const msa_config& c, const WsView& v, const void* idx_q,
                               const void* idx_k, float* scores, cudaStream_t s);
// Index scores of a decode / verify step on the tensor cores (TMA-fed tiles;
// index_score_tc.cu).
msa_status decode_index_score_tc(const msa_config& c, const WsView& v, const void* idx_q,
                                 const void* idx_k, float* scores, cudaStream_t s);
int sm_count();  // SMs of the current device (cached per device)

// Launch-status helper: any launch error becomes MSA_ERR_CUDA.
inline msa_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

// Every kernel of the path is launched with programmatic stream serialization
// (PDL): its launch and CTA start-up overlap the previous kernel's tail, and
// the kernel itself calls griddep_wait() before touching anything the previous
// kernel may still be writing or reading.  Capturable in CUDA graphs.
template <typename... KArgs, typename... Args>
inline msa_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kernel, std::forward<Args>(args)...) == cudaSuccess
             ? MSA_OK
             : MSA_ERR_CUDA;
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

// ---------------------------------------------------------------- device
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void set_error(WsHeader* h, int bits) { atomicOr(&h->err, bits); }

}  // namespace msa
