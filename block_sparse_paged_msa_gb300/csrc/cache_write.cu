// msa_cache_write: the fused K / V / index-key cache write that precedes
// attention.
//
// sglang minimax_sparse_backend.py (MiniMaxSparseAttnBackend.forward_decode and
// forward_extend) calls set_fused_kv_index_buffer(layer, out_cache_loc, k, v,
// idx_k, idx_v) before the sparse op: every new token's key, value and index
// key land in the paged pools first, which is why seq_lens already counts the
// new tokens when the index scores and the attention run.  Here the slot of a
// token is either given (out_cache_loc, sglang's page * P + row slot ids) or
// derived from the step's plan: token i of request r sits at position
// seq_len - q_len + i, i.e. row pos % P of the page the validated block table
// maps block pos / P to.
//
// Design: byte movement only.  One warp per (token, KV head): lanes 0-15 carry
// the K row and lanes 16-31 the V row (16 bytes of bf16 each), then the index
// key row and the index-value row; bf16 pools take the bytes as they are, e4m3
// pools store
// round-to-nearest-even(x / scale) codes, saturated to +-448 (NaN stays NaN),
// computed with one IEEE fp32 division and the hardware conversion.  A slot
// outside the pool is skipped and flagged (MSA_DEVERR_PAGE_RANGE), never
// written.
//
// NVFP4 pools (vLLM sparse_attention_msa.py, MiniMaxM3SparseMSANvfp4Backend:
// per KV head a key slot 2h and a value slot 2h + 1, each 72-byte row 64 bytes
// of E2M1 pairs then 8 E4M3 block scales) are written by the format's usual
// quantiser, which the pages do not spell out: a 16-element block takes the
// E4M3 code of amax / (6 * tensor scale) -- its largest magnitude onto E2M1's
// largest, 6 -- and each element the E2M1 code of x / (block scale * tensor
// scale); every step round-to-nearest-even in fp32, a block whose scale code
// is 0 stores zero codes.  A lane holds 8 elements, so a block is a lane pair.
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "msa_device.cuh"

namespace msa {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ uint4 ld_nc(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Two bf16 (one 32-bit word) -> two e4m3 codes of x / scale (low value in the
// low byte).
__device__ __forceinline__ uint32_t bf16x2_to_e4m3x2(uint32_t w, float scale) {
  const float2 f = make_float2(__fdiv_rn(bf16lo(w), scale), __fdiv_rn(bf16hi(w), scale));
  return (uint32_t)__nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
}

// Eight bf16 (this lane's part of a 16-element block; the partner lane, lane ^ 1,
// holds the rest) -> four bytes of E2M1 pairs (even element in the low nibble)
// and the block's E4M3 scale code, for tensor scale g.
__device__ __forceinline__ uint32_t nvfp4_quantize8(const uint4& x, float g, uint8_t& scale) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  float f[8], amax = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16lo(w[i]);
    f[2 * i + 1] = bf16hi(w[i]);
    amax = fmaxf(amax, fmaxf(fabsf(f[2 * i]), fabsf(f[2 * i + 1])));
  }
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  const __nv_fp8_storage_t sc =
      __nv_cvt_float_to_fp8(__fdiv_rn(amax, __fmul_rn(6.f, g)), __NV_SATFINITE, __NV_E4M3);
  scale = (uint8_t)sc;
  const float d = __fmul_rn(__half2float(__half(__nv_cvt_fp8_to_halfraw(sc, __NV_E4M3))), g);
  if (d == 0.f) return 0u;
  uint32_t codes = 0u;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 u = make_float2(__fdiv_rn(f[2 * i], d), __fdiv_rn(f[2 * i + 1], d));
    codes |= (uint32_t)__nv_cvt_float2_to_fp4x2(u, __NV_E2M1, cudaRoundNearest) << (8 * i);
  }
  return codes;
}

// kv: the pools' MSA_KV_* type.  The K and V pools may be one allocation (NVFP4
// keeps both slots of a head in every pool), hence no __restrict__ on them.
__global__ void __launch_bounds__(kWarps * 32)
cache_write_kernel(WsView ws, int Hkv, int max_blocks, int64_t pool_slots, int idx_lanes,
                   int kv, float k_scale, float v_scale, const int64_t* __restrict__ loc,
                   const uint4* __restrict__ k, const uint4* __restrict__ v,
                   const uint4* __restrict__ idx_k, const uint4* __restrict__ idx_v,
                   uint8_t* k_pages, uint8_t* v_pages,
                   uint4* __restrict__ idx_pages, uint4* __restrict__ idx_v_pages) {
  const int lane = threadIdx.x & 31;
  const int64_t item = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);   // (token, head)
  griddep_launch_dependents();
  griddep_wait();            // the plan of this step, and readers of the last one
  if (item >= (int64_t)ws.hdr->num_tokens * Hkv) return;
  const int t = (int)(item / Hkv), h = (int)(item % Hkv);
  const int r = ws.tok_req[t];
  if (r < 0) return;         // idle request: nothing to store
  int64_t slot;
  if (loc != nullptr) {
    slot = loc[t];
  } else {
    const int pos = ws.tok_pos[t];
    const int page = ws.block_table[(int64_t)r * max_blocks + pos / kBlock];
    slot = page < 0 ? -1 : (int64_t)page * kBlock + pos % kBlock;
  }
  if (slot < 0 || slot >= pool_slots) {
    if (lane == 0) set_error(ws.hdr, MSA_DEVERR_PAGE_RANGE);
    return;
  }
  // destination row in the [pages * H_kv * P] view of a pool
  const int64_t row = (slot / kBlock * Hkv + h) * kBlock + slot % kBlock;
  const int half = lane >> 4, c = lane & 15;
  const uint4 x = ld_nc((half ? v : k) + item * 16 + c);
  uint8_t* pool = half ? v_pages : k_pages;
  if (kv == MSA_KV_BF16) {
    reinterpret_cast<uint4*>(pool)[row * 16 + c] = x;
  } else if (kv == MSA_KV_NVFP4) {
    // slot 2h (keys) or 2h + 1 (values) of the page, 72-byte rows
    const int64_t r4 = ((slot / kBlock * Hkv + h) * 2 + half) * kBlock + slot % kBlock;
    uint8_t* dst = pool + r4 * kFp4Row;
    uint8_t scale;
    const uint32_t codes = nvfp4_quantize8(x, half ? v_scale : k_scale, scale);
    reinterpret_cast<uint32_t*>(dst)[c] = codes;
    if ((c & 1) == 0) dst[kHeadDim / 2 + c / 2] = scale;
  } else {
    const float s = half ? v_scale : k_scale;
    const uint32_t lo = bf16x2_to_e4m3x2(x.x, s) | bf16x2_to_e4m3x2(x.y, s) << 16;
    const uint32_t hi = bf16x2_to_e4m3x2(x.z, s) | bf16x2_to_e4m3x2(x.w, s) << 16;
    reinterpret_cast<uint2*>(pool)[row * 16 + c] = make_uint2(lo, hi);
  }
  if (idx_k != nullptr && lane < idx_lanes)
    idx_pages[row * idx_lanes + lane] = ld_nc(idx_k + item * idx_lanes + lane);
  if (idx_v != nullptr && lane < idx_lanes)
    idx_v_pages[row * idx_lanes + lane] = ld_nc(idx_v + item * idx_lanes + lane);
  // the step's later kernels read these rows with TMA (async proxy)
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" msa_status msa_cache_write(const msa_config* cfg, void* ws,
                                      const int64_t* out_cache_loc, const void* k,
                                      const void* v, const void* idx_k, const void* idx_v,
                                      void* k_pages, void* v_pages, void* idx_k_pages,
                                      void* idx_v_pages, msa_stream_t stream) {
  msa_status st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (!ws || !k || !v || !k_pages || !v_pages || (idx_k != nullptr && idx_k_pages == nullptr) ||
      (idx_v != nullptr && idx_v_pages == nullptr))
    return MSA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_pages) || !aligned16(v_pages) ||
      (idx_k && (!aligned16(idx_k) || !aligned16(idx_k_pages))) ||
      (idx_v && (!aligned16(idx_v) || !aligned16(idx_v_pages))))
    return MSA_ERR_INVALID_ARG;
  const int64_t items = (int64_t)max_tokens_of(*cfg) * cfg->num_kv_heads;
  if (items <= 0) return MSA_OK;
  const int64_t grid = (items + kWarps - 1) / kWarps;
  if (grid > 0x7fffffff) return MSA_ERR_UNSUPPORTED;
  const bool scaled = cfg->kv_dtype != MSA_KV_BF16;
  return launch_pdl(cache_write_kernel, dim3((unsigned)grid), dim3(kWarps * 32), 0,
                    (cudaStream_t)stream, view_of(*cfg, ws), cfg->num_kv_heads,
                    cfg->max_blocks_per_req, (int64_t)cfg->num_pages * kBlock,
                    cfg->index_dim / 8, (int)cfg->kv_dtype, scaled ? cfg->k_scale : 1.f,
                    scaled ? cfg->v_scale : 1.f, out_cache_loc, (const uint4*)k, (const uint4*)v,
                    (const uint4*)idx_k, (const uint4*)idx_v, (uint8_t*)k_pages,
                    (uint8_t*)v_pages, (uint4*)idx_k_pages, (uint4*)idx_v_pages);
}
