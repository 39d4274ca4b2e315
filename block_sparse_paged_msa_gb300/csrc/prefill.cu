// Chunked-prefill path: index scores for every query token of the chunk, the
// key-block -> query CSR, and block-sparse attention tiles per CSR row.
//
// vLLM minimax_m3/nvidia/sparse_attention_msa.py (MiniMaxM3SparseMSAImpl.forward)
// runs prefill as build_k2q_csr(prefill_topk [H, tokens, MK], cu_seqlens_q,
// cu_seqlens_k, block 128, total_rows, qhead_per_kv) followed by
// sparse_atten_func(q, k_cache, v_cache, row_ptr, q_indices, topK, blk_kv = 128,
// causal = True, page_table, seqused_k, ...): one dense tile per selected key
// block, causal inside the diagonal block.  sglang minimax_sparse_backend.py
// (MiniMaxSparseAttnBackend.forward_extend) feeds the same op idx_q / the
// index-K cache, cu_seqlens and prefix lengths.
//
// Here:
//  * prefill_score_kernel: a 64-token query tile x one 128-key block is a
//    dense [64 x d] x [d x 128] contraction (m16n8k16 bf16 MMA, fp32
//    accumulation, exact for integer-valued index vectors), followed by a
//    causal row max; K tiles stream through a double-buffered smem ring.
//  * csr_rows_kernel: one warp per CSR row (KV head, request, key block) walks
//    the request's tokens in order and tests membership in each token's
//    ascending selected list (binary search); ballots give the count (first
//    pass) and the ordered positions (second pass), so every row lists its
//    tokens ascending and the structure is deterministic.
//  * prefill_attn_kernel: one CTA per CSR row keeps the block's K and V tiles
//    (64 KiB) in shared memory and streams the row's tokens through it, 16
//    rows (tokens x GQA heads) per warp: S = Q K^T (bf16), causal mask, softmax
//    over the block's 128 keys, O = P V (fp16: P keeps 11 significant bits; the
//    V tile is converted once per CTA), then a normalised fp16 partial and its
//    LSE per (token, query head, slot).  msa_combine merges the slots.
#include <mutex>

#include "msa_device.cuh"

namespace msa {
namespace {

// ------------------------------------------------------------ index scores
constexpr int kScoreTokens = 64;
constexpr int kScoreThreads = 128;

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

template <int DIDX>
__device__ __forceinline__ uint32_t swz_idx(int row, int c) {
  return DIDX == 128 ? swz(row, c) : swz128(row, c);
}

template <int DIDX>
__global__ void __launch_bounds__(kScoreThreads)
prefill_score_kernel(WsView ws, int Hkv, int max_blocks, const __nv_bfloat16* __restrict__ idx_q,
                     const uint8_t* __restrict__ idx_k, float* __restrict__ scores) {
  constexpr int kRowBytes = DIDX * 2;
  constexpr int kChunks = kRowBytes / 16;
  constexpr int kTile = kBlock * kRowBytes;
  constexpr int KS = DIDX / 16;
  extern __shared__ __align__(128) uint8_t smem[];   // two K tiles
  __shared__ int seg_r[kScoreTokens + 1], seg_start[kScoreTokens + 1];
  __shared__ int nseg_s;
  griddep_launch_dependents();
  griddep_wait();
  const int T = ws.hdr->num_tokens;
  const int t0 = blockIdx.x * kScoreTokens;
  const int h = blockIdx.y;
  if (t0 >= T) return;
  const int t1 = min(T, t0 + kScoreTokens);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tq = lane & 3;
  if (tid == 0) {   // runs of consecutive tokens of one request
    int n = 0;
    for (int t = t0; t < t1; ++t) {
      const int r = ws.tok_req[t];
      if (n == 0 || r != seg_r[n - 1]) {
        seg_r[n] = r;
        seg_start[n] = t;
        ++n;
      }
    }
    seg_start[n] = t1;
    nseg_s = n;
  }
  __syncthreads();
  const int nseg = nseg_s;
  const int rowA = t0 + warp * 16 + g, rowB = rowA + 8;
  for (int sg = 0; sg < nseg; ++sg) {
    const int r = seg_r[sg];
    if (r < 0) continue;                       // CTA-uniform
    const int a = seg_start[sg], b = seg_start[sg + 1];
    const bool inA = rowA >= a && rowA < b, inB = rowB >= a && rowB < b;
    const int pA = inA ? ws.tok_pos[rowA] : -1, pB = inB ? ws.tok_pos[rowB] : -1;
    const int nblk = ws.tok_pos[b - 1] / kBlock + 1;
    uint32_t qa[KS][4];
    {
      const __nv_bfloat16* qA = idx_q + ((int64_t)rowA * Hkv + h) * DIDX;
      const __nv_bfloat16* qB = idx_q + ((int64_t)rowB * Hkv + h) * DIDX;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int c0 = ks * 16 + 2 * tq, c1 = c0 + 8;
        qa[ks][0] = inA ? ld_u32(qA + c0) : 0u;
        qa[ks][1] = inB ? ld_u32(qB + c0) : 0u;
        qa[ks][2] = inA ? ld_u32(qA + c1) : 0u;
        qa[ks][3] = inB ? ld_u32(qB + c1) : 0u;
      }
    }
    auto issue = [&](int j, int buf) {
      const int page = ws.block_table[(int64_t)r * max_blocks + j];
      const uint8_t* src = idx_k + ((int64_t)(page < 0 ? 0 : page) * Hkv + h) * (int64_t)kTile;
      const uint32_t dst = smem_u32(smem + buf * kTile);
#pragma unroll
      for (int k = 0; k < kBlock * kChunks / kScoreThreads; ++k) {
        const int idx = k * kScoreThreads + tid;
        const int row = idx / kChunks, c = idx % kChunks;
        cp_async16(dst + swz_idx<DIDX>(row, c), src + row * kRowBytes + c * 16, page < 0 ? 0 : 16);
      }
      cp_async_commit();
    };
    issue(0, 0);
    for (int j = 0; j < nblk; ++j) {
      if (j + 1 < nblk) issue(j + 1, (j + 1) & 1); else cp_async_commit();
      cp_async_wait<1>();
      __syncthreads();
      const uint32_t tile = smem_u32(smem + (j & 1) * kTile);
      float mA = -INFINITY, mB = -INFINITY;
#pragma unroll 4
      for (int nt = 0; nt < 16; ++nt) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        const int krow = nt * 8 + (lane & 7);
#pragma unroll
        for (int ks = 0; ks < KS; ks += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(tile + swz_idx<DIDX>(krow, 2 * ks + (lane >> 3)), b0, b1, b2, b3);
          mma_bf16(c, qa[ks], b0, b1);
          mma_bf16(c, qa[ks + 1], b2, b3);
        }
        const int key = j * kBlock + nt * 8 + 2 * tq;
        if (key <= pA) mA = fmaxf(mA, c[0]);
        if (key + 1 <= pA) mA = fmaxf(mA, c[1]);
        if (key <= pB) mB = fmaxf(mB, c[2]);
        if (key + 1 <= pB) mB = fmaxf(mB, c[3]);
      }
      mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, 1));
      mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, 2));
      mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, 1));
      mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, 2));
      if (tq == 0) {
        if (inA && j * kBlock <= pA) scores[((int64_t)rowA * Hkv + h) * max_blocks + j] = mA;
        if (inB && j * kBlock <= pB) scores[((int64_t)rowB * Hkv + h) * max_blocks + j] = mB;
      }
      __syncthreads();
    }
    cp_async_wait<0>();
  }
}

// ------------------------------------------------------------ CSR
__device__ __forceinline__ bool has_block(const int32_t* sel, int n, int j) {
  int lo = 0, hi = n;            // sel[0..n) ascending
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (sel[mid] < j) lo = mid + 1; else hi = mid;
  }
  return lo < n && sel[lo] == j;
}

template <bool FILL>
__global__ void __launch_bounds__(256)
csr_rows_kernel(WsView ws, int Hkv, int B, int NB, int S, const int32_t* __restrict__ selected,
                int32_t* __restrict__ row_ptr, int32_t* __restrict__ q_idx) {
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  griddep_launch_dependents();
  griddep_wait();
  if (row >= (int64_t)Hkv * B * NB) return;
  const int j = (int)(row % NB);
  const int r = (int)((row / NB) % B);
  const int h = (int)(row / ((int64_t)NB * B));
  int count = 0;
  const int base = FILL ? row_ptr[row] : 0;
  if (r < ws.hdr->batch && j < ws.req_nb[r]) {
    const int qs = ws.req_qstart[r], qe = ws.req_qstart[r + 1];
    for (int t0 = qs; t0 < qe; t0 += 32) {
      const int t = t0 + lane;
      bool in = false;
      if (t < qe && ws.tok_req[t] == r) {
        const int p = ws.tok_pos[t];
        if (j * kBlock <= p) {
          const int n = min(p / kBlock + 1, S);
          in = has_block(selected + ((int64_t)t * Hkv + h) * S, n, j);
        }
      }
      const unsigned bal = __ballot_sync(0xffffffffu, in);
      if (FILL && in) q_idx[base + count + __popc(bal & ((1u << lane) - 1u))] = t;
      count += __popc(bal);
    }
  }
  if (!FILL && lane == 0) {
    row_ptr[row + 1] = count;
    if (row == 0) row_ptr[0] = 0;
  }
}

// In-place inclusive scan of row_ptr[1..rows] (one CTA: each thread owns a
// contiguous segment; a block scan of the segment sums gives the offsets).
__global__ void __launch_bounds__(1024) csr_scan_kernel(int32_t* __restrict__ row_ptr, int64_t rows) {
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  griddep_launch_dependents();
  griddep_wait();
  const int64_t seg = (rows + 1023) / 1024;
  const int64_t lo = tid * seg, hi = min(rows, lo + seg);
  int sum = 0;
  for (int64_t k = lo; k < hi; ++k) sum += row_ptr[1 + k];
  int x = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += warp_tot[w];
  int run = before + x - sum;
  for (int64_t k = lo; k < hi; ++k) {
    run += row_ptr[1 + k];
    row_ptr[1 + k] = run;
  }
}

// ------------------------------------------------------------ attention
constexpr int kPfThreads = 256;
constexpr int kTileBytes = kBlock * kHeadDim * 2;

struct PrefillArgs {
  int Hkv, Hq, G, S, B, NB;
  float scale_log2;
  const __nv_bfloat16* q;
  const uint8_t* k;
  const uint8_t* v;
  const int32_t* selected;
  const int32_t* row_ptr;
  const int32_t* q_idx;
};

__device__ __forceinline__ int slot_of(const int32_t* sel, int n, int j) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (sel[mid] < j) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kPfThreads, 1)
prefill_attn_kernel(WsView ws, PrefillArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];   // K tile, V tile
  griddep_launch_dependents();
  griddep_wait();
  const int64_t row = blockIdx.x;
  const int j = (int)(row % a.NB);
  const int r = (int)((row / a.NB) % a.B);
  const int h = (int)(row / ((int64_t)a.NB * a.B));
  const int beg = a.row_ptr[row], end = a.row_ptr[row + 1];
  if (beg >= end) return;
  const int page = ws.block_table[(int64_t)r * a.NB + j];
  if (page < 0) return;
  const int ntok = min(kBlock, ws.req_seq_len[r] - j * kBlock);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tq = lane & 3;
  {
    const uint32_t dst = smem_u32(smem);
#pragma unroll
    for (int kind = 0; kind < 2; ++kind) {
      const uint8_t* src = (kind == 0 ? a.k : a.v) +
                           ((int64_t)page * a.Hkv + h) * (int64_t)kTileBytes;
#pragma unroll
      for (int k = 0; k < kBlock * 16 / kPfThreads; ++k) {
        const int idx = k * kPfThreads + tid;
        const int rr = idx >> 4, c = idx & 15;
        const bool ok = rr < ntok;
        cp_async16(dst + kind * kTileBytes + swz(rr, c), src + (ok ? rr * 256 + c * 16 : 0),
                   ok ? 16 : 0);
      }
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    // V to fp16 in place: P V runs as an fp16 MMA, so the probabilities keep
    // 11 significant bits instead of bf16's 8.
    uint4* vt = reinterpret_cast<uint4*>(smem + kTileBytes);
    for (int i = tid; i < kTileBytes / 16; i += kPfThreads) {
      uint4 w = vt[i];
      w.x = bf16x2_to_f16x2(w.x); w.y = bf16x2_to_f16x2(w.y);
      w.z = bf16x2_to_f16x2(w.z); w.w = bf16x2_to_f16x2(w.w);
      vt[i] = w;
    }
    __syncthreads();
  }
  const uint32_t ktile = smem_u32(smem), vtile = ktile + kTileBytes;
  const int TPW = kMaxGroup / a.G;                 // tokens per warp per pass
  const int lt0 = warp * TPW + g / a.G, lt1 = warp * TPW + (g + 8) / a.G;
  const int hg0 = g % a.G, hg1 = (g + 8) % a.G;
  for (int base = beg; base < end; base += 8 * TPW) {
    const int i0 = base + lt0, i1 = base + lt1;
    const bool v0 = i0 < end, v1 = i1 < end;
    const int t_0 = v0 ? a.q_idx[i0] : 0, t_1 = v1 ? a.q_idx[i1] : 0;
    const int p0 = v0 ? ws.tok_pos[t_0] : -1, p1 = v1 ? ws.tok_pos[t_1] : -1;
    uint32_t qa[8][4];
    {
      const __nv_bfloat16* q0 = a.q + ((int64_t)t_0 * a.Hq + h * a.G + hg0) * kHeadDim;
      const __nv_bfloat16* q1 = a.q + ((int64_t)t_1 * a.Hq + h * a.G + hg1) * kHeadDim;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int c0 = ks * 16 + 2 * tq, c1 = c0 + 8;
        qa[ks][0] = v0 ? ld_u32(q0 + c0) : 0u;
        qa[ks][1] = v1 ? ld_u32(q1 + c0) : 0u;
        qa[ks][2] = v0 ? ld_u32(q0 + c1) : 0u;
        qa[ks][3] = v1 ? ld_u32(q1 + c1) : 0u;
      }
    }
    float sc[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
      const int krow = nt * 8 + (lane & 7);
#pragma unroll
      for (int ks = 0; ks < 8; ks += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(ktile + swz(krow, 2 * ks + (lane >> 3)), b0, b1, b2, b3);
        mma_bf16(sc[nt], qa[ks], b0, b1);
        mma_bf16(sc[nt], qa[ks + 1], b2, b3);
      }
    }
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = nt * 8 + 2 * tq + (e & 1);
        const int p = e < 2 ? p0 : p1;
        const bool ok = key < ntok && j * kBlock + key <= p;
        sc[nt][e] = ok ? sc[nt][e] * a.scale_log2 : -INFINITY;
        if (e < 2) m0 = fmaxf(m0, sc[nt][e]); else m1 = fmaxf(m1, sc[nt][e]);
      }
    }
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
    const float mr0 = m0 == -INFINITY ? 0.f : m0, mr1 = m1 == -INFINITY ? 0.f : m1;
    float l0 = 0.f, l1 = 0.f;
    uint32_t pa[8][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const __half2 h01 = __floats2half2_rn(exp2f(sc[nt][0] - mr0), exp2f(sc[nt][1] - mr0));
      const __half2 h23 = __floats2half2_rn(exp2f(sc[nt][2] - mr1), exp2f(sc[nt][3] - mr1));
      const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
      l0 += f01.x + f01.y;            // normalise by the probabilities actually used
      l1 += f23.x + f23.y;
      pa[nt >> 1][(nt & 1) * 2 + 0] = *reinterpret_cast<const uint32_t*>(&h01);
      pa[nt >> 1][(nt & 1) * 2 + 1] = *reinterpret_cast<const uint32_t*>(&h23);
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    float o[16][4];
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int vrow = kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
      for (int nd = 0; nd < 16; nd += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vtile + swz(vrow, nd + (lane >> 4)), b0, b1, b2, b3);
        mma_f16(o[nd], pa[kk], b0, b1);
        mma_f16(o[nd + 1], pa[kk], b2, b3);
      }
    }
    // normalised fp16 partial + LSE for (token, head, slot of j)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const bool ok = half == 0 ? v0 : v1;
      if (!ok) continue;
      const int t = half == 0 ? t_0 : t_1;
      const int p = half == 0 ? p0 : p1;
      const int hq = h * a.G + (half == 0 ? hg0 : hg1);
      const float l = half == 0 ? l0 : l1;
      const float m = half == 0 ? m0 : m1;
      const int nsel = min(p / kBlock + 1, a.S);
      const int slot = slot_of(a.selected + ((int64_t)t * a.Hkv + h) * a.S, nsel, j);
      if (slot >= nsel) continue;                  // j not selected: cannot happen for a CSR entry
      const int64_t pi = ((int64_t)t * a.Hq + hq) * a.S + slot;
      __half* op = static_cast<__half*>(ws.o_part) + pi * kHeadDim;
      const float inv = 1.f / l;
#pragma unroll
      for (int nd = 0; nd < 16; ++nd) {
        const float x0 = o[nd][half * 2] * inv, x1 = o[nd][half * 2 + 1] * inv;
        *reinterpret_cast<uint32_t*>(op + nd * 8 + 2 * tq) = pack_f16(x0, x1);
      }
      if (tq == 0) ws.lse_part[pi] = (m + log2f(l)) * kLn2;
    }
  }
}

template <typename K>
msa_status set_smem(K kernel, size_t bytes) {
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) ==
                 cudaSuccess
             ? MSA_OK
             : MSA_ERR_CUDA;
}

}  // namespace

msa_status prefill_index_score(const msa_config& c, const WsView& v, const void* idx_q,
                               const void* idx_k, float* scores, cudaStream_t s) {
  const int T = max_tokens_of(c);
  dim3 grid((T + kScoreTokens - 1) / kScoreTokens, c.num_kv_heads);
  const size_t smem = 2u * kBlock * c.index_dim * 2;
  msa_status st;
  if (c.index_dim == 128) {
    if ((st = set_smem(prefill_score_kernel<128>, smem)) != MSA_OK) return st;
    return launch_pdl(prefill_score_kernel<128>, grid, dim3(kScoreThreads), smem, s, v,
                      c.num_kv_heads, c.max_blocks_per_req, (const __nv_bfloat16*)idx_q,
                      (const uint8_t*)idx_k, scores);
  }
  if ((st = set_smem(prefill_score_kernel<64>, smem)) != MSA_OK) return st;
  return launch_pdl(prefill_score_kernel<64>, grid, dim3(kScoreThreads), smem, s, v,
                    c.num_kv_heads, c.max_blocks_per_req, (const __nv_bfloat16*)idx_q,
                    (const uint8_t*)idx_k, scores);
}

}  // namespace msa

using namespace msa;

extern "C" int64_t msa_k2q_rows(const msa_config* cfg) {
  return check_config(cfg) == MSA_OK ? csr_rows_of(*cfg) : 0;
}

extern "C" int64_t msa_k2q_capacity(const msa_config* cfg) {
  return check_config(cfg) == MSA_OK
             ? (int64_t)max_tokens_of(*cfg) * cfg->num_kv_heads * width_of(*cfg)
             : 0;
}

extern "C" msa_status msa_build_k2q_csr(const msa_config* cfg, const void* ws,
                                        const int32_t* selected, int32_t* row_ptr,
                                        int32_t* q_indices, msa_stream_t stream) {
  msa_status st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (!is_prefill(*cfg)) return MSA_ERR_INVALID_ARG;
  if (!ws || !selected || !row_ptr || !q_indices) return MSA_ERR_INVALID_ARG;
  const int64_t rows = csr_rows_of(*cfg);
  if (rows + 1 > 0x7fffffff || (rows + 7) / 8 > 0x7fffffff) return MSA_ERR_UNSUPPORTED;
  const WsView v = view_of(*cfg, ws);
  cudaStream_t s = (cudaStream_t)stream;
  const unsigned grid = (unsigned)((rows + 7) / 8);
  const int S = width_of(*cfg);
  if ((st = launch_pdl(csr_rows_kernel<false>, dim3(grid), dim3(256), 0, s, v, cfg->num_kv_heads,
                       cfg->max_batch, cfg->max_blocks_per_req, S, selected, row_ptr,
                       q_indices)) != MSA_OK)
    return st;
  if ((st = launch_pdl(csr_scan_kernel, dim3(1), dim3(1024), 0, s, row_ptr, rows)) != MSA_OK)
    return st;
  return launch_pdl(csr_rows_kernel<true>, dim3(grid), dim3(256), 0, s, v, cfg->num_kv_heads,
                    cfg->max_batch, cfg->max_blocks_per_req, S, selected, row_ptr, q_indices);
}

extern "C" msa_status msa_sparse_prefill(const msa_config* cfg, void* ws, const void* q,
                                         const void* k_pages, const void* v_pages,
                                         const int32_t* selected, const int32_t* row_ptr,
                                         const int32_t* q_indices, msa_stream_t stream) {
  msa_status st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (!is_prefill(*cfg)) return MSA_ERR_INVALID_ARG;
  if (cfg->kv_dtype != MSA_KV_BF16) return MSA_ERR_UNSUPPORTED;
  if (!ws || !q || !k_pages || !v_pages || !selected || !row_ptr || !q_indices)
    return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages)) return MSA_ERR_INVALID_ARG;
  const int64_t rows = csr_rows_of(*cfg);
  if (rows > 0x7fffffff) return MSA_ERR_UNSUPPORTED;
  PrefillArgs a;
  a.Hkv = cfg->num_kv_heads;
  a.Hq = cfg->num_q_heads;
  a.G = cfg->num_q_heads / cfg->num_kv_heads;
  a.S = width_of(*cfg);
  a.B = cfg->max_batch;
  a.NB = cfg->max_blocks_per_req;
  a.scale_log2 = cfg->softmax_scale * kLog2e;
  a.q = (const __nv_bfloat16*)q;
  a.k = (const uint8_t*)k_pages;
  a.v = (const uint8_t*)v_pages;
  a.selected = selected;
  a.row_ptr = row_ptr;
  a.q_idx = q_indices;
  const size_t smem = 2u * kTileBytes;
  if ((st = set_smem(prefill_attn_kernel, smem)) != MSA_OK) return st;
  return launch_pdl(prefill_attn_kernel, dim3((unsigned)rows), dim3(kPfThreads), smem,
                    (cudaStream_t)stream, view_of(*cfg, ws), a);
}
