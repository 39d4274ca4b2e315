// msa_sparse_decode + msa_combine: split-K flash decoding over the selected
// blocks of a paged KV cache, then a log-sum-exp merge of the splits.
//
// vLLM minimax_m3/nvidia/sparse_attention_msa.py (module docstring and
// MiniMaxM3SparseMSAImpl.forward) runs decode as a split-K kernel over the
// top-k blocks, with block_table, seq_lens and decode_query_len, and
// dequantises fp8 KV on load with per-layer k/v scales; sglang
// minimax_sparse_backend.py (MiniMaxSparseAttnBackend.forward_decode) passes
// the query, the K/V cache and the per-request page table to the same op.
//
// Work item = (query token t, KV head h, split s); a split is a run of
// consecutive slots of t's selected list.  One 128-thread CTA per item:
//  * the G = H_q / H_kv query heads of h form the M side of an m16n8k16 bf16
//    MMA (rows >= G are zero), the group shares every K/V tile it loads;
//  * each selected block contributes a 32 KiB K tile and a 32 KiB V tile
//    ([128 tokens][128 dims], contiguous per page and head in the HND pool),
//    staged through a 3-deep ring of shared-memory tiles with 16-byte
//    cp.async copies (XOR-swizzled 16-byte chunks so that ldmatrix reads are
//    conflict-free; rows past the last visible token are zero-filled, never
//    read);
//  * warp w owns tokens [32w, 32w+32) of every tile and keeps its own online
//    softmax state; the four states are merged once at the end of the item;
//  * fp8-e4m3 tiles (16 KiB) are converted to bf16 in shared memory (e4m3 is
//    exact in bf16); k_scale is folded into the softmax scale and v_scale into
//    the output.
// The partial output (normalised) and its natural-log LSE go to the workspace;
// msa_combine merges them in a fixed order (deterministic).
#include <mutex>

#include "msa_device.cuh"

namespace msa {
namespace {

constexpr int kThreads = 128;
constexpr int kStages = 3;
constexpr int kTileBytes = kBlock * kHeadDim * 2;  // bf16 tile, 32 KiB

struct DecodeArgs {
  int Hkv, Hq, G, S, bps, nsplit, max_blocks;
  float scale_log2;     // softmax_scale * k_scale * log2(e)
  float v_scale;
  const __nv_bfloat16* q;
  const uint8_t* k;     // bf16 or e4m3 pool
  const uint8_t* v;
  const int32_t* selected;
};

// Issue the copy of one K or V tile (block slot i, kind 0 = K, 1 = V) into ring
// buffer `buf`.  bf16: 2048 16-byte chunks, swizzled.  fp8: 1024 raw chunks.
template <bool FP8>
__device__ __forceinline__ void issue_tile(const DecodeArgs& a, uint8_t* ring, int buf,
                                           int page, int h, int ntok, int kind) {
  const uint8_t* pool = kind == 0 ? a.k : a.v;
  constexpr int kRowBytes = FP8 ? 128 : 256;
  constexpr int kChunksPerRow = kRowBytes / 16;
  const uint8_t* src = pool + ((int64_t)page * a.Hkv + h) * (int64_t)kBlock * kRowBytes;
  uint8_t* dst = ring + buf * kTileBytes;
  const uint32_t dst_s = smem_u32(dst);
#pragma unroll
  for (int k = 0; k < kBlock * kChunksPerRow / kThreads; ++k) {
    const int idx = k * kThreads + threadIdx.x;
    const int row = idx / kChunksPerRow, c = idx % kChunksPerRow;
    const int bytes = row < ntok ? 16 : 0;                // zero-fill past the end
    const uint8_t* g = src + (row < ntok ? row * kRowBytes + c * 16 : 0);
    const uint32_t off = FP8 ? (uint32_t)(row * kRowBytes + c * 16) : swz(row, c);
    cp_async16(dst_s + off, g, bytes);
  }
}

// fp8: convert the raw tile at the start of ring buffer `buf` into the bf16
// swizzled tile `conv`.
__device__ __forceinline__ void convert_tile(const uint8_t* raw, uint8_t* conv) {
#pragma unroll
  for (int k = 0; k < (kBlock * 8) / kThreads; ++k) {       // 1024 raw chunks
    const int idx = k * kThreads + threadIdx.x;
    const int row = idx >> 3, c = idx & 7;
    const uint4 w = *reinterpret_cast<const uint4*>(raw + row * 128 + c * 16);
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t o[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      o[2 * e] = e4m3x2_to_bf16x2((uint16_t)(in[e] & 0xffffu));
      o[2 * e + 1] = e4m3x2_to_bf16x2((uint16_t)(in[e] >> 16));
    }
    *reinterpret_cast<uint4*>(conv + swz(row, 2 * c)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(conv + swz(row, 2 * c + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

template <bool FP8>
__global__ void __launch_bounds__(kThreads)
decode_kernel(WsView ws, DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;                                     // kStages tiles
  uint8_t* conv = smem + kStages * kTileBytes;              // fp8: bf16 staging tile
  __shared__ int blk_page[64], blk_ntok[64];
  __shared__ int n_blk_s;
  __shared__ float red_m[4][16], red_l[4][16];

  const int item = blockIdx.x;
  const int s = item % a.nsplit;
  const int h = (item / a.nsplit) % a.Hkv;
  const int t = item / (a.nsplit * a.Hkv);
  if (t >= ws.hdr->num_tokens) return;
  const int r = ws.tok_req[t];
  if (r < 0) return;                                        // combine writes 0 / -inf
  const int pos = ws.tok_pos[t];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tq = lane & 3;

  // ---- the split's blocks: (page, visible rows), invalid slots dropped
  if (tid < 32) {
    const int slot0 = s * a.bps;
    const int nslot = min(a.bps, a.S - slot0);
    int page = -1, ntok = 0;
    if (lane < nslot) {
      const int j = a.selected[((int64_t)t * a.Hkv + h) * a.S + slot0 + lane];
      if (j >= 0 && j * kBlock <= pos) {
        page = ws.block_table[(int64_t)r * a.max_blocks + j];
        ntok = min(kBlock, pos + 1 - j * kBlock);
      }
    }
    const bool ok = page >= 0 && lane < nslot;
    const unsigned bal = __ballot_sync(0xffffffffu, ok);
    if (ok) {
      const int p = __popc(bal & ((1u << lane) - 1u));
      blk_page[p] = page;
      blk_ntok[p] = ntok;
    }
    if (lane == 0) n_blk_s = __popc(bal);
  }
  // ---- Q fragments (rows = query heads of the group, zero past G)
  uint32_t qa[8][4];
  {
    const __nv_bfloat16* qb = a.q + ((int64_t)t * a.Hq + (int64_t)h * a.G) * kHeadDim;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int c0 = ks * 16 + 2 * tq, c1 = c0 + 8;
      qa[ks][0] = g < a.G ? *reinterpret_cast<const uint32_t*>(qb + g * kHeadDim + c0) : 0u;
      qa[ks][1] = g + 8 < a.G ? *reinterpret_cast<const uint32_t*>(qb + (g + 8) * kHeadDim + c0) : 0u;
      qa[ks][2] = g < a.G ? *reinterpret_cast<const uint32_t*>(qb + g * kHeadDim + c1) : 0u;
      qa[ks][3] = g + 8 < a.G ? *reinterpret_cast<const uint32_t*>(qb + (g + 8) * kHeadDim + c1) : 0u;
    }
  }
  __syncthreads();
  const int nblk = n_blk_s;
  const int ntiles = 2 * nblk;   // K0 V0 K1 V1 ...

  float acc[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY};   // running max (log2 domain), rows g, g+8
  float l_r[2] = {0.f, 0.f};               // per-thread partial row sums
  uint32_t pa[2][4];                        // P as bf16 A fragments (2 k-steps)

  // ---- prologue
#pragma unroll
  for (int x = 0; x < kStages - 1; ++x) {
    if (x < ntiles) issue_tile<FP8>(a, ring, x, blk_page[x >> 1], h, blk_ntok[x >> 1], x & 1);
    cp_async_commit();
  }
  for (int x = 0; x < ntiles; ++x) {
    {
      const int y = x + kStages - 1;
      if (y < ntiles) issue_tile<FP8>(a, ring, y % kStages, blk_page[y >> 1], h, blk_ntok[y >> 1], y & 1);
      cp_async_commit();
    }
    cp_async_wait<kStages - 1>();
    __syncthreads();
    const uint8_t* tile = ring + (x % kStages) * kTileBytes;
    if (FP8) {
      convert_tile(tile, conv);
      __syncthreads();
      tile = conv;
    }
    const uint32_t tile_s = smem_u32(tile);
    const int ntok = blk_ntok[x >> 1];
    if ((x & 1) == 0) {
      // ---- S = Q K^T for this warp's 32 tokens (4 n-tiles of 8)
      float sc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
        const int row = warp * 32 + nt * 8 + (lane & 7);
#pragma unroll
        for (int ks = 0; ks < 8; ks += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(tile_s + swz(row, 2 * ks + (lane >> 3)), b0, b1, b2, b3);
          mma_bf16(sc[nt], qa[ks], b0, b1);
          mma_bf16(sc[nt], qa[ks + 1], b2, b3);
        }
      }
      // ---- online softmax (log2 domain), rows g (c0,c1) and g+8 (c2,c3)
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int tok = warp * 32 + nt * 8 + 2 * tq;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool valid = tok + (e & 1) < ntok;
          sc[nt][e] = valid ? sc[nt][e] * a.scale_log2 : -INFINITY;
          mx[e >> 1] = fmaxf(mx[e >> 1], sc[nt][e]);
        }
      }
      float alpha[2], mref[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
        mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
        const float mn = fmaxf(m_r[i], mx[i]);
        mref[i] = mn == -INFINITY ? 0.f : mn;
        alpha[i] = exp2f(m_r[i] - mref[i]);
        m_r[i] = mn;
        l_r[i] *= alpha[i];
      }
#pragma unroll
      for (int nd = 0; nd < 16; ++nd) {
        acc[nd][0] *= alpha[0]; acc[nd][1] *= alpha[0];
        acc[nd][2] *= alpha[1]; acc[nd][3] *= alpha[1];
      }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p = exp2f(sc[nt][e] - mref[e >> 1]);
          sc[nt][e] = p;
          l_r[e >> 1] += p;
        }
      }
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        pa[kk][0] = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
        pa[kk][1] = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
        pa[kk][2] = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
        pa[kk][3] = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
      }
    } else {
      // ---- O += P V for this warp's 32 tokens (2 k-steps of 16)
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int row = warp * 32 + kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
        for (int nd = 0; nd < 16; nd += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(tile_s + swz(row, nd + (lane >> 4)), b0, b1, b2, b3);
          mma_bf16(acc[nd], pa[kk], b0, b1);
          mma_bf16(acc[nd + 1], pa[kk], b2, b3);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  // ---- merge the four warps' states
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l_r[i] += __shfl_xor_sync(0xffffffffu, l_r[i], 1);
    l_r[i] += __shfl_xor_sync(0xffffffffu, l_r[i], 2);
  }
  if (tq == 0) {
    red_m[warp][g] = m_r[0];
    red_m[warp][g + 8] = m_r[1];
    red_l[warp][g] = l_r[0];
    red_l[warp][g + 8] = l_r[1];
  }
  __syncthreads();
  float* red = reinterpret_cast<float*>(smem);   // [4 warps][16 rows][128] fp32, 32 KiB
  float fw[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int row = g + 8 * i;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, red_m[w][row]);
    fw[i] = M == -INFINITY ? 0.f : exp2f(m_r[i] - M);
  }
#pragma unroll
  for (int nd = 0; nd < 16; ++nd) {
    const int col = nd * 8 + 2 * tq;
    float* p0 = red + (warp * 16 + g) * kHeadDim + col;
    float* p1 = red + (warp * 16 + g + 8) * kHeadDim + col;
    *reinterpret_cast<float2*>(p0) = make_float2(acc[nd][0] * fw[0], acc[nd][1] * fw[0]);
    *reinterpret_cast<float2*>(p1) = make_float2(acc[nd][2] * fw[1], acc[nd][3] * fw[1]);
  }
  __syncthreads();
  // thread = output column; rows < G
  const int col = tid;
  for (int row = 0; row < a.G; ++row) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, red_m[w][row]);
    float L = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float f = M == -INFINITY ? 0.f : exp2f(red_m[w][row] - M);
      L += red_l[w][row] * f;
      o += red[(w * 16 + row) * kHeadDim + col];
    }
    const int64_t hq = (int64_t)t * a.Hq + (int64_t)h * a.G + row;
    const bool empty = !(L > 0.f);
    static_cast<float*>(ws.o_part)[(hq * a.nsplit + s) * kHeadDim + col] =
        empty ? 0.f : o * (a.v_scale / L);
    if (col == 0)
      ws.lse_part[hq * a.nsplit + s] = empty ? -INFINITY : (M + log2f(L)) * kLn2;
  }
}

// ---- combine: one warp per (token, query head), splits merged in a fixed
// order.  PREFILL: fp16 partials, one per selected slot, of which the first
// min(nb, S) exist (nb = the token's visible blocks).
template <bool PREFILL>
__global__ void __launch_bounds__(256)
combine_kernel(WsView ws, int Hq, int nsplit, __nv_bfloat16* __restrict__ out,
               float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int64_t idx = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int t = (int)(idx / Hq);
  if (t >= ws.hdr->num_tokens) return;
  const bool active = ws.tok_req[t] >= 0;
  int nvalid = nsplit;
  if (PREFILL) nvalid = active ? min(nsplit, ws.tok_pos[t] / kBlock + 1) : 0;
  const float* lp = ws.lse_part + idx * nsplit;
  float M = -INFINITY;
  if (active)
    for (int s = lane; s < nvalid; s += 32) M = fmaxf(M, lp[s]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    float L = 0.f;
    for (int s = 0; s < nvalid; ++s) L += exp2f((lp[s] - M) * kLog2e);
    const float lse_tot = M + logf(L);
    for (int s = 0; s < nvalid; ++s) {
      const float w = expf(lp[s] - lse_tot);
      float4 v;
      if (PREFILL) {
        const uint2 raw = *reinterpret_cast<const uint2*>(
            static_cast<const __half*>(ws.o_part) + (idx * nsplit + s) * kHeadDim + 4 * lane);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
        v = make_float4(a.x, a.y, b.x, b.y);
      } else {
        v = *reinterpret_cast<const float4*>(static_cast<const float*>(ws.o_part) +
                                             (idx * nsplit + s) * kHeadDim + 4 * lane);
      }
      o.x = fmaf(w, v.x, o.x); o.y = fmaf(w, v.y, o.y);
      o.z = fmaf(w, v.z, o.z); o.w = fmaf(w, v.w, o.w);
    }
    if (lane == 0) lse[idx] = lse_tot;
  } else if (lane == 0) {
    lse[idx] = -INFINITY;
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y), hi = __floats2bfloat162_rn(o.z, o.w);
  uint2 pk = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  *reinterpret_cast<uint2*>(out + idx * kHeadDim + 4 * lane) = pk;
}

template <bool FP8>
size_t decode_smem() {
  return (size_t)kStages * kTileBytes + (FP8 ? kTileBytes : 0);
}

template <bool FP8>
msa_status ensure_smem_attr() {
  static std::mutex mu;
  static bool done[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return MSA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(mu);
  if (!done[dev]) {
    if (cudaFuncSetAttribute(decode_kernel<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)decode_smem<FP8>()) != cudaSuccess)
      return MSA_ERR_CUDA;
    done[dev] = true;
  }
  return MSA_OK;
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" msa_status msa_sparse_decode(const msa_config* cfg, void* ws, const void* q,
                                        const void* k_pages, const void* v_pages,
                                        const int32_t* selected, msa_stream_t stream) {
  msa_status st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (!ws || !q || !k_pages || !v_pages || !selected) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages)) return MSA_ERR_INVALID_ARG;
  if (is_prefill(*cfg)) return MSA_ERR_INVALID_ARG;   // prefill uses msa_sparse_prefill
  const int S = width_of(*cfg);
  if (S > 64 * 1024) return MSA_ERR_UNSUPPORTED;
  DecodeArgs a;
  a.Hkv = cfg->num_kv_heads;
  a.Hq = cfg->num_q_heads;
  a.G = cfg->num_q_heads / cfg->num_kv_heads;
  a.S = S;
  a.bps = blocks_per_split_of(*cfg);
  if (a.bps > 32) return MSA_ERR_UNSUPPORTED;   // one warp lists a split's blocks
  a.nsplit = splits_of(*cfg);
  a.max_blocks = cfg->max_blocks_per_req;
  const bool fp8 = cfg->kv_dtype == MSA_KV_FP8_E4M3;
  a.scale_log2 = cfg->softmax_scale * (fp8 ? cfg->k_scale : 1.f) * kLog2e;
  a.v_scale = fp8 ? cfg->v_scale : 1.f;
  a.q = (const __nv_bfloat16*)q;
  a.k = (const uint8_t*)k_pages;
  a.v = (const uint8_t*)v_pages;
  a.selected = selected;
  const int64_t grid = (int64_t)max_tokens_of(*cfg) * a.Hkv * a.nsplit;
  if (grid <= 0) return MSA_OK;
  if (grid > 0x7fffffff) return MSA_ERR_UNSUPPORTED;
  const WsView v = view_of(*cfg, ws);
  cudaStream_t s = (cudaStream_t)stream;
  if (fp8) {
    if ((st = ensure_smem_attr<true>()) != MSA_OK) return st;
    decode_kernel<true><<<(unsigned)grid, kThreads, decode_smem<true>(), s>>>(v, a);
  } else {
    if ((st = ensure_smem_attr<false>()) != MSA_OK) return st;
    decode_kernel<false><<<(unsigned)grid, kThreads, decode_smem<false>(), s>>>(v, a);
  }
  return launch_status();
}

extern "C" msa_status msa_combine(const msa_config* cfg, const void* ws, void* out, float* lse,
                                  msa_stream_t stream) {
  msa_status st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (!ws || !out || !lse) return MSA_ERR_INVALID_ARG;
  if (((uintptr_t)out & 7) != 0) return MSA_ERR_INVALID_ARG;
  const int64_t items = (int64_t)max_tokens_of(*cfg) * cfg->num_q_heads;
  if (items <= 0) return MSA_OK;
  const int64_t grid = (items + 7) / 8;
  if (grid > 0x7fffffff) return MSA_ERR_UNSUPPORTED;
  if (is_prefill(*cfg))
    combine_kernel<true><<<(unsigned)grid, 256, 0, (cudaStream_t)stream>>>(
        view_of(*cfg, ws), cfg->num_q_heads, splits_of(*cfg), (__nv_bfloat16*)out, lse);
  else
    combine_kernel<false><<<(unsigned)grid, 256, 0, (cudaStream_t)stream>>>(
        view_of(*cfg, ws), cfg->num_q_heads, splits_of(*cfg), (__nv_bfloat16*)out, lse);
  return launch_status();
}
