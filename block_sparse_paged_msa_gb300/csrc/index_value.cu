// msa_index_attention: the index-value branch's output idx_o.
//
// sglang minimax_sparse_backend.py keeps, for the layers outside
// disable_value_layer_ids, an index-value cache beside the index keys
// (MiniMaxSparseAttnBackend.get_index_kv_buffer, written with idx_v by
// set_fused_kv_index_buffer), and the sparse decode / prefill ops return
// (idx_o, o) with idx_o of shape [tokens, num_idx_heads * idx_head_dim].  The
// pages do not give idx_o's formula.  This library reads the index head as a
// dense causal attention head over every visible token:
//   idx_o[t, h] = softmax_u(idx_q[t, h] . idx_k[u, h] / sqrt(d)) idx_v[u, h],
//   u over the request's tokens at positions <= position(t),
// i.e. the same dot products the index scores take their block maxima of.
//
// Design: split-K over each token's visible blocks, like the decode.  A warp
// per (token, KV head, split of consecutive blocks): the lanes own 16-byte
// slices of the index dimension (d / 8 lanes per key row, 32 / (d / 8) rows
// per warp-wide load), a row's dot product is reduced across its lanes, and
// each row group keeps its own online softmax (exp2 domain) over chunks of 8
// rows before the groups merge; the partial (max, sum, unnormalised output)
// goes to the caller's scratch.  A second kernel merges a token's splits in
// a fixed order.
#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kIvWarps = 8;
constexpr int kIvSplitsMax = 32;
constexpr int kIvUnroll = 8;       // rows per group per chunk: its key and value rows are
                                   // requested together (16 16-byte loads in flight per lane)

inline int iv_splits(const msa_config& c) {
  return c.max_blocks_per_req < kIvSplitsMax ? c.max_blocks_per_req : kIvSplitsMax;
}
inline int iv_blocks_per_split(const msa_config& c) {
  const int ns = iv_splits(c);
  return (c.max_blocks_per_req + ns - 1) / ns;
}

__device__ __forceinline__ uint4 ld_stream16(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void unpack8(const uint4& w, float (&f)[8]) {
  f[0] = bf16lo(w.x); f[1] = bf16hi(w.x);
  f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
  f[4] = bf16lo(w.z); f[5] = bf16hi(w.z);
  f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
}

template <int DIDX>
__global__ void __launch_bounds__(kIvWarps * 32)
index_attn_partial_kernel(WsView ws, int Hkv, int max_blocks, int NS, int bps, float scale_log2,
                          const uint4* __restrict__ idx_q, const uint4* __restrict__ idx_k,
                          const uint4* __restrict__ idx_v, float* __restrict__ o_part,
                          float2* __restrict__ ml_part) {
  constexpr int LPR = DIDX / 8;         // lanes per key row
  constexpr int RPI = 32 / LPR;         // row groups (rows per warp-wide load)
  const int lane = threadIdx.x & 31, sub = lane % LPR, grp = lane / LPR;
  const int64_t item = (int64_t)blockIdx.x * kIvWarps + (threadIdx.x >> 5);   // (t, h, split)
  griddep_launch_dependents();
  griddep_wait();
  if (item >= (int64_t)ws.hdr->num_tokens * Hkv * NS) return;                // warp-uniform
  const int s = (int)(item % NS), h = (int)((item / NS) % Hkv), t = (int)(item / ((int64_t)NS * Hkv));
  float m = -INFINITY, l = 0.f, o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  const int r = ws.tok_req[t];
  if (r >= 0) {
    const int pos = ws.tok_pos[t];
    const int nb = pos / kBlock + 1;
    const int jb = s * bps, je = min(nb, jb + bps);
    float q[8];
    unpack8(idx_q[(((int64_t)t * Hkv + h) * DIDX) / 8 + sub], q);
    for (int j = jb; j < je; ++j) {
      const int page = ws.block_table[(int64_t)r * max_blocks + j];   // warp-uniform
      if (page < 0) continue;                                          // flagged by the plan
      const int lim = min(kBlock, pos + 1 - j * kBlock);               // visible rows
      const int64_t base = (((int64_t)page * Hkv + h) * kBlock * DIDX) / 8;
#pragma unroll 1
      for (int rb = 0; rb < kBlock; rb += RPI * kIvUnroll) {
        // the chunk's key and value rows in flight together (a value row past
        // the token's position is read from the page but never used)
        uint4 kr[kIvUnroll], vr[kIvUnroll];
#pragma unroll
        for (int u = 0; u < kIvUnroll; ++u) {
          const int64_t at = base + (rb + u * RPI + grp) * LPR + sub;
          kr[u] = ld_stream16(idx_k + at);
          vr[u] = ld_stream16(idx_v + at);
        }
        float sc[kIvUnroll];
#pragma unroll
        for (int u = 0; u < kIvUnroll; ++u) {
          const int row = rb + u * RPI + grp;
          float k8[8];
          unpack8(kr[u], k8);
          float x = q[0] * k8[0];
#pragma unroll
          for (int i = 1; i < 8; ++i) x = fmaf(q[i], k8[i], x);
#pragma unroll
          for (int msk = 1; msk < LPR; msk <<= 1) x += __shfl_xor_sync(0xffffffffu, x, msk);
          sc[u] = row < lim ? x * scale_log2 : -INFINITY;
        }
        float cm = sc[0];
#pragma unroll
        for (int u = 1; u < kIvUnroll; ++u) cm = fmaxf(cm, sc[u]);
        const float mn = fmaxf(m, cm);
        const float alpha = mn == -INFINITY ? 1.f : exp2f(m - mn);
        l *= alpha;
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] *= alpha;
        m = mn;
#pragma unroll
        for (int u = 0; u < kIvUnroll; ++u) {
          if (sc[u] == -INFINITY) continue;   // rows past the position: not used
          const float p = exp2f(sc[u] - mn);
          float v8[8];
          unpack8(vr[u], v8);
          l += p;
#pragma unroll
          for (int i = 0; i < 8; ++i) o[i] = fmaf(p, v8[i], o[i]);
        }
      }
    }
  }
  // merge the row groups' states (same d-slice in lanes sub, sub + LPR, ...)
#pragma unroll
  for (int msk = LPR; msk < 32; msk <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, msk);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, msk);
    const float mn = fmaxf(m, m2);
    const float a1 = mn == -INFINITY ? 0.f : exp2f(m - mn);
    const float a2 = mn == -INFINITY ? 0.f : exp2f(m2 - mn);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float o2 = __shfl_xor_sync(0xffffffffu, o[i], msk);
      o[i] = o[i] * a1 + o2 * a2;
    }
    l = l * a1 + l2 * a2;
    m = mn;
  }
  if (grp == 0) {
    float4* dst = reinterpret_cast<float4*>(o_part + item * DIDX + sub * 8);
    dst[0] = make_float4(o[0], o[1], o[2], o[3]);
    dst[1] = make_float4(o[4], o[5], o[6], o[7]);
    if (sub == 0) ml_part[item] = make_float2(m, l);
  }
}

// Merge of a token's splits, in split order: warp per (token, KV head), lane
// owning d / 32 output values.
template <int DIDX>
__global__ void __launch_bounds__(256)
index_attn_combine_kernel(WsView ws, int Hkv, int NS, const float* __restrict__ o_part,
                          const float2* __restrict__ ml_part, __nv_bfloat16* __restrict__ out,
                          float* __restrict__ lse) {
  constexpr int VPL = DIDX / 32;        // values per lane
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);   // (t, h)
  griddep_launch_dependents();
  griddep_wait();
  if (row >= (int64_t)ws.hdr->num_tokens * Hkv) return;
  const int t = (int)(row / Hkv);
  const float2* ml = ml_part + row * NS;
  float M = -INFINITY;
  if (ws.tok_req[t] >= 0)
    for (int s = lane; s < NS; s += 32) M = fmaxf(M, ml[s].x);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float acc[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) acc[i] = 0.f;
  float L = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < NS; ++s) {
      const float2 x = ml[s];
      if (x.y <= 0.f) continue;
      const float w = exp2f(x.x - M);
      L += x.y * w;
      const float* op = o_part + (row * NS + s) * DIDX + lane * VPL;
#pragma unroll
      for (int i = 0; i < VPL; ++i) acc[i] = fmaf(w, op[i], acc[i]);
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16* dst = out + row * DIDX + lane * VPL;
#pragma unroll
  for (int i = 0; i < VPL; ++i) dst[i] = __float2bfloat16_rn(acc[i] * inv);
  if (lse != nullptr && lane == 0) lse[row] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

template <int DIDX>
msa_status launch_iv(const msa_config& c, const WsView& v, const void* idx_q, const void* idx_k,
                     const void* idx_v, void* scratch, void* out, float* lse, cudaStream_t s) {
  const int NS = iv_splits(c), bps = iv_blocks_per_split(c);
  const int64_t rows = (int64_t)max_tokens_of(c) * c.num_kv_heads;
  const int64_t items = rows * NS;
  if ((items + kIvWarps - 1) / kIvWarps > 0x7fffffff) return MSA_ERR_UNSUPPORTED;
  float* o_part = static_cast<float*>(scratch);
  float2* ml_part = reinterpret_cast<float2*>(static_cast<char*>(scratch) +
                                              align_up((size_t)items * DIDX * 4));
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)DIDX);
  msa_status st = launch_pdl(index_attn_partial_kernel<DIDX>,
                             dim3((unsigned)((items + kIvWarps - 1) / kIvWarps)),
                             dim3(kIvWarps * 32), 0, s, v, c.num_kv_heads, c.max_blocks_per_req,
                             NS, bps, scale_log2, (const uint4*)idx_q, (const uint4*)idx_k,
                             (const uint4*)idx_v, o_part, ml_part);
  if (st != MSA_OK) return st;
  return launch_pdl(index_attn_combine_kernel<DIDX>, dim3((unsigned)((rows + 7) / 8)), dim3(256),
                    0, s, v, c.num_kv_heads, NS, (const float*)o_part, (const float2*)ml_part,
                    (__nv_bfloat16*)out, lse);
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" size_t msa_index_attention_scratch_bytes(const msa_config* cfg) {
  if (check_config(cfg) != MSA_OK || is_prefill(*cfg)) return 0;
  const size_t items = (size_t)max_tokens_of(*cfg) * cfg->num_kv_heads * iv_splits(*cfg);
  return align_up(items * cfg->index_dim * 4) + align_up(items * 8);
}

extern "C" msa_status msa_index_attention(const msa_config* cfg, const void* ws, const void* idx_q,
                                          const void* idx_k_pages, const void* idx_v_pages,
                                          void* scratch, void* idx_out, float* idx_lse,
                                          msa_stream_t stream) {
  msa_status st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (is_prefill(*cfg)) return MSA_ERR_UNSUPPORTED;
  if (!ws || !idx_q || !idx_k_pages || !idx_v_pages || !scratch || !idx_out)
    return MSA_ERR_INVALID_ARG;
  if (!aligned16(idx_q) || !aligned16(idx_k_pages) || !aligned16(idx_v_pages) ||
      ((uintptr_t)scratch & 255) != 0 || ((uintptr_t)idx_out & 3) != 0)
    return MSA_ERR_INVALID_ARG;
  if (max_tokens_of(*cfg) * (int64_t)cfg->num_kv_heads <= 0) return MSA_OK;
  const WsView v = view_of(*cfg, ws);
  cudaStream_t s = (cudaStream_t)stream;
  return cfg->index_dim == 128
             ? launch_iv<128>(*cfg, v, idx_q, idx_k_pages, idx_v_pages, scratch, idx_out, idx_lse, s)
             : launch_iv<64>(*cfg, v, idx_q, idx_k_pages, idx_v_pages, scratch, idx_out, idx_lse, s);
}
