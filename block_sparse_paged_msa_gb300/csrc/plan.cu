// msa_plan: per-step metadata built on the device, plus the host-side ABI
// helpers (status strings, config checks, workspace sizing, error readback).
//
// The plan follows the metadata the serving backends prepare before attention:
// sglang MiniMaxSparseAttnBackend._prepare_msa_decode_meta builds a decode plan
// per batch size outside graph capture and refreshes a kv-indices buffer from
// req_to_token / req_pool_indices / seq_lens in place; vLLM
// MiniMaxM3SparseMSAMetadataBuilder.build hands block_table, seq_lens and
// decode_query_len to the decode kernel.  Here everything is derived on the
// device into a fixed-shape workspace so that a captured graph can replay it.
#include <cuda.h>

#include <mutex>
#include <vector>

#include "msa_internal.cuh"

namespace msa {

int32_t blocks_per_split_of(const msa_config& c) {
  const int32_t S = width_of(c);
  if (S <= 0) return 1;
  if (c.blocks_per_split > 0) return c.blocks_per_split < S ? c.blocks_per_split : S;
  // The decode kernel is persistent (two CTAs per SM) and streams across item
  // boundaries, so items only need to outnumber the CTAs: aim for about 512
  // (fewer, longer items mean fewer partials to merge; measured flat from 2
  // to 20 blocks per item on the medium decode workload), at most 32 blocks
  // per item (one warp lists an item's blocks).
  const int64_t items = (int64_t)max_tokens_of(c) * c.num_kv_heads;
  int64_t ns = items > 0 ? (512 + items - 1) / items : 1;
  if (ns < 1) ns = 1;
  if (ns > S) ns = S;
  int32_t bps = (int32_t)((S + ns - 1) / ns);
  if (bps > 32) bps = (S + (S + 31) / 32 - 1) / ((S + 31) / 32);
  return bps;
}

msa_status check_config(const msa_config* c) {
  if (c == nullptr) return MSA_ERR_INVALID_ARG;
  if (c->num_q_heads <= 0 || c->num_kv_heads <= 0 || c->init_blocks < 0 ||
      c->local_blocks < 1 || c->topk_blocks < 0 || c->q_len < 1 || c->max_batch < 0 ||
      c->max_q_tokens < 0 || c->max_blocks_per_req < 1 || c->num_pages < 1 ||
      c->blocks_per_split < 0 || !(c->softmax_scale > 0.f))
    return MSA_ERR_INVALID_ARG;
  if (c->num_q_heads % c->num_kv_heads != 0) return MSA_ERR_INVALID_ARG;
  if (c->kv_dtype != MSA_KV_BF16 && c->kv_dtype != MSA_KV_FP8_E4M3 &&
      c->kv_dtype != MSA_KV_NVFP4)
    return MSA_ERR_INVALID_ARG;
  if (c->kv_dtype != MSA_KV_BF16 && !(c->k_scale > 0.f && c->v_scale > 0.f))
    return MSA_ERR_INVALID_ARG;
  if (c->head_dim != kHeadDim || c->block_size != kBlock) return MSA_ERR_UNSUPPORTED;
  if (c->index_dim != 64 && c->index_dim != 128) return MSA_ERR_UNSUPPORTED;
  if (c->num_q_heads / c->num_kv_heads > kMaxGroup) return MSA_ERR_UNSUPPORTED;
  if (c->mode != MSA_MODE_DECODE && c->mode != MSA_MODE_PREFILL) return MSA_ERR_INVALID_ARG;
  if (c->mode == MSA_MODE_PREFILL && (kMaxGroup % (c->num_q_heads / c->num_kv_heads)) != 0)
    return MSA_ERR_UNSUPPORTED;
  if (c->mode == MSA_MODE_PREFILL && c->max_q_tokens <= 0) return MSA_ERR_INVALID_ARG;
  if (c->max_blocks_per_req > kMaxBlocksPerReq || c->max_batch > kMaxBatch)
    return MSA_ERR_UNSUPPORTED;
  if ((int64_t)max_tokens_of(*c) * c->num_q_heads > (int64_t)1 << 30) return MSA_ERR_UNSUPPORTED;
  return MSA_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool make_bf16_map(CUtensorMap* m, const void* base, int rank, const int64_t* dims,
                   const int64_t* strides_bytes, const int* box) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], estr[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = (cuuint64_t)dims[i];
    bx[i] = (cuuint32_t)box[i];
    estr[i] = 1u;
    if (i > 0) st[i - 1] = (cuuint64_t)strides_bytes[i - 1];
  }
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), d, st,
             bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_pool_map(CUtensorMap* m, const void* base, int64_t rows, bool fp8, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * (fp8 ? 1 : 2)};
  const cuuint32_t box[2] = {fp8 ? 128u : 64u, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
             const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

// ----------------------------------------------------------------- kernels
struct ReqInfo {
  bool valid;
  int L, nq, qs, nb;
};

// Validates request r.  seq_len 0 is an idle request (no tokens, no error).
__device__ __forceinline__ ReqInfo request_info(int r, const int* seq_lens, const int* cu_q,
                                                int q_len, int max_blocks, int max_tokens) {
  ReqInfo ri;
  const int L = seq_lens[r];
  const int qs = cu_q ? cu_q[r] : r * q_len;
  const int qe = cu_q ? cu_q[r + 1] : (r + 1) * q_len;
  ri.qs = qs;
  ri.nq = qe - qs;
  ri.L = L;
  ri.valid = L > 0 && L <= max_blocks * kBlock && qs >= 0 && ri.nq >= 0 && ri.nq <= L &&
             qe <= max_tokens;
  ri.nb = ri.valid ? (L + kBlock - 1) / kBlock : 0;
  return ri;
}

__device__ __forceinline__ bool request_flagged(int r, const int* seq_lens, const int* cu_q,
                                                int q_len, int max_blocks, int max_tokens) {
  ReqInfo ri = request_info(r, seq_lens, cu_q, q_len, max_blocks, max_tokens);
  return !ri.valid && !(ri.L == 0);
}

// One CTA per request copies (and validates) its block-table row; CTA 0 also
// builds the request / token metadata.
__global__ void __launch_bounds__(256)
plan_kernel(WsView ws, int batch, int max_batch, int Hkv, int q_len, int max_blocks,
            int max_tokens, int num_pages, const int* __restrict__ seq_lens,
            const int* __restrict__ cu_q, const int* __restrict__ bt, int bt_stride,
            const int* __restrict__ r2t, int r2t_stride, const int64_t* __restrict__ pool_idx) {
  const int tid = threadIdx.x;
  const int r = blockIdx.x;
  griddep_launch_dependents();
  griddep_wait();            // the previous step may still read this workspace
  if (r == 0 && tid == 0) {
    ws.hdr->err = 0;         // later kernels' bits; this kernel reports in plan_err
    ws.hdr->max_batch = max_batch;
    ws.hdr->work_next = 0;
    ws.hdr->work_done = 0;
  }
  if (r < batch) {
    ReqInfo ri = request_info(r, seq_lens, cu_q, q_len, max_blocks, max_tokens);
    int bad = 0;
    for (int j = tid; j < ri.nb; j += blockDim.x) {
      int page;
      if (bt != nullptr) {
        page = bt[(int64_t)r * bt_stride + j];
      } else {
        const int64_t row = pool_idx[r];
        const int slot = r2t[row * r2t_stride + (int64_t)j * kBlock];
        page = slot >= 0 ? slot / kBlock : -1;
        if (slot >= 0 && slot % kBlock != 0) bad |= MSA_DEVERR_SLOT_ALIGN;
      }
      if (page < 0 || page >= num_pages) {
        bad |= MSA_DEVERR_PAGE_RANGE;
        page = -1;
      }
      ws.block_table[(int64_t)r * max_blocks + j] = page;
    }
    if (tid == 0 && request_flagged(r, seq_lens, cu_q, q_len, max_blocks, max_tokens))
      bad |= MSA_DEVERR_SEQ_LEN;
    __shared__ int bad_s;
    if (tid == 0) bad_s = 0;
    __syncthreads();
    if (bad) atomicOr(&bad_s, bad);
    __syncthreads();
    if (tid == 0) ws.plan_err[r] = bad_s;
  }
  if (r != 0) return;
  for (int i = (batch > 0 ? batch : 0) + tid; i < (max_batch > 0 ? max_batch : 1); i += blockDim.x)
    ws.plan_err[i] = 0;

  // ---- CTA 0: per-request block counts and prefix sums (chunked block scan)
  __shared__ int warp_sums[8];
  __shared__ int carry_s;
  if (tid == 0) carry_s = 0;
  __syncthreads();
  const int lane = tid & 31, warp = tid >> 5;
  for (int base = 0; base < batch; base += blockDim.x) {
    const int rr = base + tid;
    int nb = 0;
    if (rr < batch) {
      ReqInfo ri = request_info(rr, seq_lens, cu_q, q_len, max_blocks, max_tokens);
      nb = ri.nb;
      ws.req_seq_len[rr] = ri.valid ? ri.L : 0;
      ws.req_nb[rr] = nb;
      ws.req_qstart[rr] = ri.qs;
    }
    int x = nb;  // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    int before = carry_s;
    for (int w = 0; w < warp; ++w) before += warp_sums[w];
    if (rr < batch) ws.req_cu_nb[rr] = before + x - nb;
    __syncthreads();
    if (tid == 0) {
      int tot = 0;
      for (int w = 0; w < 8; ++w) tot += warp_sums[w];
      carry_s += tot;
    }
    __syncthreads();
  }
  int T = 0;
  if (batch > 0) {
    T = cu_q ? cu_q[batch] : batch * q_len;
    if (T < 0) T = 0;
    if (T > max_tokens) {
      T = max_tokens;
      if (tid == 0) set_error(ws.hdr, MSA_DEVERR_SEQ_LEN);   // after the reset above
    }
  }
  if (tid == 0) {
    ws.req_cu_nb[batch] = carry_s;
    ws.req_qstart[batch] = T;
    ws.hdr->batch = batch;
    ws.hdr->num_tokens = T;
    ws.hdr->total_blocks = carry_s;
  }
  // ---- per-token (request, position); tokens of no valid request stay -1
  for (int t = tid; t < max_tokens; t += blockDim.x) {
    ws.tok_req[t] = -1;
    ws.tok_pos[t] = -1;
  }
  __syncthreads();
  for (int rr = warp; rr < batch; rr += blockDim.x / 32) {
    ReqInfo ri = request_info(rr, seq_lens, cu_q, q_len, max_blocks, max_tokens);
    if (!ri.valid) continue;
    for (int i = lane; i < ri.nq; i += 32) {
      ws.tok_req[ri.qs + i] = rr;
      ws.tok_pos[ri.qs + i] = ri.L - ri.nq + i;
    }
  }
}

static msa_status plan_common(const msa_config* cfg, int32_t batch, const int32_t* seq_lens,
                              const int32_t* cu_q, const int32_t* bt, int32_t bt_stride,
                              const int32_t* r2t, int32_t r2t_stride, const int64_t* pool_idx,
                              void* ws, msa_stream_t stream) {
  msa_status st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (ws == nullptr || ((uintptr_t)ws & 255) != 0) return MSA_ERR_INVALID_ARG;
  if (batch < 0 || batch > cfg->max_batch) return MSA_ERR_INVALID_ARG;
  if (batch > 0 && seq_lens == nullptr) return MSA_ERR_INVALID_ARG;
  if (batch > 0 && bt == nullptr && (r2t == nullptr || pool_idx == nullptr))
    return MSA_ERR_INVALID_ARG;
  if (bt != nullptr && bt_stride < cfg->max_blocks_per_req) return MSA_ERR_INVALID_ARG;
  if (cfg->mode == MSA_MODE_PREFILL && batch > 0 && cu_q == nullptr) return MSA_ERR_INVALID_ARG;
  if (r2t != nullptr && r2t_stride < cfg->max_blocks_per_req * kBlock) return MSA_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  WsView v = view_of(*cfg, ws);
  return launch_pdl(plan_kernel, dim3(batch > 0 ? batch : 1), dim3(256), 0, s, v, batch,
                    cfg->max_batch, cfg->num_kv_heads, cfg->q_len, cfg->max_blocks_per_req,
                    max_tokens_of(*cfg), cfg->num_pages, seq_lens, cu_q, bt, bt_stride, r2t,
                    r2t_stride, pool_idx);
}

}  // namespace msa

using namespace msa;

extern "C" {

const char* msa_status_string(msa_status s) {
  switch (s) {
    case MSA_OK: return "MSA_OK";
    case MSA_ERR_INVALID_ARG: return "MSA_ERR_INVALID_ARG: invalid argument";
    case MSA_ERR_UNSUPPORTED: return "MSA_ERR_UNSUPPORTED: configuration not implemented";
    case MSA_ERR_CUDA: return "MSA_ERR_CUDA: a CUDA runtime call failed";
    case MSA_ERR_DEVICE_FLAG: return "MSA_ERR_DEVICE_FLAG: a kernel flagged invalid data";
  }
  return "unknown msa_status";
}

msa_status msa_validate_config(const msa_config* cfg) { return check_config(cfg); }

int32_t msa_init_blocks_from_tokens(int32_t tokens, int32_t block_size) {
  if (tokens < 0 || block_size <= 0) return -1;
  return (int32_t)(((int64_t)tokens + block_size - 1) / block_size);
}

int32_t msa_local_blocks_from_tokens(int32_t tokens, int32_t block_size) {
  if (tokens < 0 || block_size <= 0) return -1;
  return (int32_t)(((int64_t)tokens + block_size - 1) / block_size + 1);
}

int32_t msa_selected_width(const msa_config* cfg) {
  return check_config(cfg) == MSA_OK ? width_of(*cfg) : 0;
}

int32_t msa_num_splits(const msa_config* cfg) {
  return check_config(cfg) == MSA_OK ? splits_of(*cfg) : 0;
}

size_t msa_workspace_bytes(const msa_config* cfg) {
  if (check_config(cfg) != MSA_OK) return 0;
  return layout_of(*cfg).total;
}

msa_status msa_plan(const msa_config* cfg, int32_t batch, const int32_t* seq_lens,
                    const int32_t* cu_seqlens_q, const int32_t* block_table, int32_t bt_stride,
                    void* ws, msa_stream_t stream) {
  if (batch > 0 && block_table == nullptr) return MSA_ERR_INVALID_ARG;
  return plan_common(cfg, batch, seq_lens, cu_seqlens_q, block_table, bt_stride, nullptr, 0,
                     nullptr, ws, stream);
}

msa_status msa_plan_from_req_to_token(const msa_config* cfg, int32_t batch,
                                      const int32_t* seq_lens, const int32_t* cu_seqlens_q,
                                      const int32_t* req_to_token, int32_t r2t_stride,
                                      const int64_t* req_pool_indices, void* ws,
                                      msa_stream_t stream) {
  if (batch > 0 && (req_to_token == nullptr || req_pool_indices == nullptr))
    return MSA_ERR_INVALID_ARG;
  return plan_common(cfg, batch, seq_lens, cu_seqlens_q, nullptr, 0, req_to_token, r2t_stride,
                     req_pool_indices, ws, stream);
}

msa_status msa_check_device_error(const void* ws, int32_t* flags, msa_stream_t stream) {
  if (ws == nullptr || flags == nullptr) return MSA_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  WsHeader h;
  if (cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MSA_ERR_CUDA;
  int32_t bits = h.err;
  const int n = h.max_batch > 0 ? h.max_batch : 1;
  if (n <= kMaxBatch) {   // the plan's per-request words follow the 256-byte header
    std::vector<int32_t> pe(n);
    if (cudaMemcpyAsync(pe.data(), (const char*)ws + 256, sizeof(int32_t) * n,
                        cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return MSA_ERR_CUDA;
    for (int32_t e : pe) bits |= e;
  }
  *flags = bits;
  return bits ? MSA_ERR_DEVICE_FLAG : MSA_OK;
}

}  // extern "C"
