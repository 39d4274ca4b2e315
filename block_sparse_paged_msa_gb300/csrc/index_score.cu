// msa_index_score: per (query token, KV head, visible block) the maximum over
// the block's visible tokens of idx_q . idx_k.
//
// sglang minimax_sparse_backend.py (MiniMaxSparseAttnBackend.__init__) reads
// the index head dim (sparse_index_dim) and a score_type, and forward_decode
// hands idx_q and the index-K cache to the sparse decode op; the score formula
// itself is fixed by this library's specification: max over tokens, fp32
// accumulation, no scale.
//
// Design (GB300): a pure HBM scan -- every visible index key is read once per
// request (one 256-byte row per token and KV head at d = 128) against 128 FMAs,
// about 0.5 FMA per byte, so CUDA cores are ample and the kernel is sized for
// bytes in flight.  One warp owns one half (64 rows) of a (block, KV head)
// tile, which is contiguous in the HND page layout (16 KiB at d = 128); the two
// halves' maxima meet in the score with an order-free atomic max over scores
// set to -inf by a first small kernel (a whole tile per warp left a tail: a
// warp took 6 or 7 tiles of ~26 us each, so the last third of them ran ~15 us
// alone).  Lanes own a fixed
// 16-byte slice of the index dimension, so the index query stays in registers;
// each lane keeps 8 16-byte streaming loads in flight, and the partial dot
// products of 8 rows are reduced across the row's lanes with a
// transpose-reduce butterfly (one shuffle per row instead of log2(lanes)).
// The grid is persistent (SMs x resident CTAs) and walks the flattened
// (request, block, head) list, so ragged sequence lengths balance by blocks,
// not by requests; a unit finds its request by a binary search over the
// requests' first blocks, or, for up to 32 requests, by one ballot over them
// kept in the warp's registers.
#include <algorithm>
#include <mutex>

#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;   // 16-byte loads in flight per lane
constexpr int kParts = 2;    // work units per (block, KV head) tile: row ranges of kBlock / kParts

// Max of a score slot and x, in any order of arrival: a non-negative float
// orders like its int bits, a negative one reversely like its unsigned bits;
// -0 is taken as +0.  The slot starts at -inf.  x is never NaN here (the
// warp's own max ignores NaN rows; a part of only NaN rows is not written).
__device__ __forceinline__ void atomic_max_score(float* slot, float x) {
  x = x + 0.0f;
  if (x >= 0.f) atomicMax(reinterpret_cast<int*>(slot), __float_as_int(x));
  else atomicMin(reinterpret_cast<unsigned int*>(slot), __float_as_uint(x));
}

// Every score slot of the step's tokens to -inf (the parts meet by atomic max).
__global__ void __launch_bounds__(256)
score_init_kernel(WsView ws, int64_t row_slots, float* __restrict__ scores) {
  griddep_launch_dependents();
  griddep_wait();
  const int64_t n = (int64_t)ws.hdr->num_tokens * row_slots;
  for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256)
    scores[i] = -INFINITY;
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float dot8(const float (&q)[8], const uint4& w) {
  float s = q[0] * bf16lo(w.x);
  s = fmaf(q[1], bf16hi(w.x), s);
  s = fmaf(q[2], bf16lo(w.y), s);
  s = fmaf(q[3], bf16hi(w.y), s);
  s = fmaf(q[4], bf16lo(w.z), s);
  s = fmaf(q[5], bf16hi(w.z), s);
  s = fmaf(q[6], bf16lo(w.w), s);
  s = fmaf(q[7], bf16hi(w.w), s);
  return s;
}

// DIDX: index dim (64 | 128).  QL: query tokens per request scored together,
// sharing every key load (instantiated for decode, QL = 1; speculative verify
// runs on the tensor-core kernel, whose tile stream does not depend on the
// q_len x d / 8 registers the queries take here).
template <int DIDX, int QL>
__global__ void __launch_bounds__(kThreads, QL == 1 ? 5 : 2)
index_score_kernel(WsView ws, int Hkv, int max_blocks, int max_tokens,
                   const uint4* __restrict__ idx_q,
                   const uint4* __restrict__ idx_k, float* __restrict__ scores) {
  constexpr int LPR = DIDX / 8;            // lanes per key row
  constexpr int RPI = 32 / LPR;            // rows per warp-wide load
  constexpr int ROWS = kUnroll * RPI;      // rows per batch
  static_assert((kBlock / kParts) % ROWS == 0, "a part must be a multiple of the batch");
  const int lane = threadIdx.x & 31;
  const int sub = lane % LPR, rsub = lane / LPR;
  // Row (within a batch) whose full dot product this lane holds after the
  // transpose-reduce: the upper-half lanes keep the upper half at every step.
  int u_lane = 0;
  {
    int n = kUnroll;
#pragma unroll
    for (int mask = LPR / 2; mask >= 1; mask >>= 1) {
      if (n > 1) {
        n >>= 1;
        if (sub & mask) u_lane += n;
      }
    }
  }
  griddep_launch_dependents();
  griddep_wait();
  const int batch = ws.hdr->batch;
  const int total = ws.hdr->total_blocks * Hkv * kParts;
  const int warps = gridDim.x * (kThreads / 32);
  // up to 32 requests: lane i keeps request i's first flat block, and a unit
  // finds its request with one ballot instead of a search through memory
  const bool small_batch = batch <= 32;
  const int cu_lane = small_batch && lane < batch ? ws.req_cu_nb[lane] : 0x7fffffff;
  for (int item = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); item < total;
       item += warps) {
    const int h = item % Hkv;
    const int part = (item / Hkv) % kParts;
    const int b = item / (Hkv * kParts);
    const int r0 = part * (kBlock / kParts);   // this unit's rows [r0, r0 + kBlock / kParts)
    int r, j;                    // request of flat block b, and its block
    if (small_batch) {
      r = __popc(__ballot_sync(0xffffffffu, cu_lane <= b)) - 1;
      j = b - __shfl_sync(0xffffffffu, cu_lane, r);
    } else {
      int lo = 0, hi = batch - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ws.req_cu_nb[mid] <= b) lo = mid; else hi = mid - 1;
      }
      r = lo;
      j = b - ws.req_cu_nb[r];
    }
    const int page = ws.block_table[(int64_t)r * max_blocks + j];
    const int qs = ws.req_qstart[r];
    float* out = scores + ((int64_t)qs * Hkv + h) * max_blocks + j;
    if (page < 0) {  // flagged by the plan; never dereferenced
      if (lane == 0)
        for (int i = 0; i < QL; ++i)
          if (qs + i < max_tokens && ws.tok_req[qs + i] == r)
            out[(int64_t)i * Hkv * max_blocks] = -INFINITY;
      continue;
    }
    float q[QL][8];
    int lim[QL];
#pragma unroll
    for (int i = 0; i < QL; ++i) {
      // a request owns QL consecutive tokens; anything else is left unscored
      const bool mine = qs + i < max_tokens && ws.tok_req[qs + i] == r;
      const uint4 w = mine ? idx_q[(((int64_t)(qs + i) * Hkv + h) * DIDX) / 8 + sub]
                           : make_uint4(0u, 0u, 0u, 0u);
      q[i][0] = bf16lo(w.x); q[i][1] = bf16hi(w.x);
      q[i][2] = bf16lo(w.y); q[i][3] = bf16hi(w.y);
      q[i][4] = bf16lo(w.z); q[i][5] = bf16hi(w.z);
      q[i][6] = bf16lo(w.w); q[i][7] = bf16hi(w.w);
      lim[i] = mine ? ws.tok_pos[qs + i] - j * kBlock + 1 : 0;  // visible rows
    }
    bool any = false;                          // a visible row in this part
#pragma unroll
    for (int i = 0; i < QL; ++i) any |= lim[i] > r0;
    if (!any) continue;
    const uint4* tile = idx_k + (((int64_t)page * Hkv + h) * kBlock * DIDX) / 8;
    float best[QL];
#pragma unroll
    for (int i = 0; i < QL; ++i) best[i] = -INFINITY;
#pragma unroll 1
    for (int rb = r0; rb < r0 + kBlock / kParts; rb += ROWS) {
      uint4 d[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) d[u] = ld_stream(tile + (rb + u * RPI + rsub) * LPR + sub);
#pragma unroll
      for (int i = 0; i < QL; ++i) {
        float v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) v[u] = dot8(q[i], d[u]);
        int n = kUnroll;
#pragma unroll
        for (int mask = LPR / 2; mask >= 1; mask >>= 1) {
          if (n > 1) {
            const int half = n >> 1;
            const bool upper = (sub & mask) != 0;
#pragma unroll
            for (int k = 0; k < half; ++k) {
              const float send = upper ? v[k] : v[k + half];
              const float keep = upper ? v[k + half] : v[k];
              v[k] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
            }
            n = half;
          } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
          }
        }
        const int row = rb + u_lane * RPI + rsub;
        if (row < lim[i]) best[i] = fmaxf(best[i], v[0]);
      }
    }
#pragma unroll
    for (int i = 0; i < QL; ++i) {
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1)
        best[i] = fmaxf(best[i], __shfl_xor_sync(0xffffffffu, best[i], o));
      if (lane == 0 && lim[i] > r0 && !isnan(best[i]))
        atomic_max_score(out + (int64_t)i * Hkv * max_blocks, best[i]);
    }
  }
}

template <int DIDX, int QL>
msa_status launch(const msa_config& c, const WsView& v, const void* idx_q, const void* idx_k,
                  float* scores, cudaStream_t s) {
  static std::mutex mu;
  static int occ[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return MSA_ERR_CUDA;
  int blocks_per_sm;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (occ[dev] == 0) {
      int n = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, index_score_kernel<DIDX, QL>,
                                                        kThreads, 0) != cudaSuccess)
        return MSA_ERR_CUDA;
      occ[dev] = n > 0 ? n : 1;
    }
    blocks_per_sm = occ[dev];
  }
  const int grid = sm_count() * blocks_per_sm;
  if (grid <= 0) return MSA_ERR_CUDA;
  const int64_t row_slots = (int64_t)c.num_kv_heads * c.max_blocks_per_req;
  const int64_t slots = (int64_t)max_tokens_of(c) * row_slots;
  const unsigned igrid = (unsigned)std::min<int64_t>((slots + 255) / 256, (int64_t)sm_count() * 8);
  msa_status st = launch_pdl(score_init_kernel, dim3(igrid > 0 ? igrid : 1), dim3(256), 0, s, v,
                             row_slots, scores);
  if (st != MSA_OK) return st;
  return launch_pdl(index_score_kernel<DIDX, QL>, dim3(grid), dim3(kThreads), 0, s, v,
                    c.num_kv_heads, c.max_blocks_per_req, max_tokens_of(c),
                    (const uint4*)idx_q, (const uint4*)idx_k, scores);
}

// One new token per request (decode); several (verify) go to the tensor-core
// kernel of index_score_tc.cu.
msa_status dispatch(const msa_config& c, const WsView& v, const void* idx_q, const void* idx_k,
                    float* scores, cudaStream_t s) {
  return c.index_dim == 128 ? launch<128, 1>(c, v, idx_q, idx_k, scores, s)
                            : launch<64, 1>(c, v, idx_q, idx_k, scores, s);
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" msa_status msa_index_score(const msa_config* cfg, const void* ws, const void* idx_q,
                                      const void* idx_k_pages, float* block_scores,
                                      msa_stream_t stream) {
  msa_status st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (!ws || !idx_q || !idx_k_pages || !block_scores) return MSA_ERR_INVALID_ARG;
  if (!aligned16(idx_q) || !aligned16(idx_k_pages)) return MSA_ERR_INVALID_ARG;
  const WsView v = view_of(*cfg, ws);
  cudaStream_t s = (cudaStream_t)stream;
  if (is_prefill(*cfg)) return prefill_index_score(*cfg, v, idx_q, idx_k_pages, block_scores, s);
  // Several new tokens per request (speculative verify) share every key tile:
  // the tensor-core kernel, whose tile stream does not depend on registers.
  if (cfg->q_len > 1) return decode_index_score_tc(*cfg, v, idx_q, idx_k_pages, block_scores, s);
  return dispatch(*cfg, v, idx_q, idx_k_pages, block_scores, s);
}

extern "C" msa_status msa_index_score_topk(const msa_config* cfg, void* ws, const void* idx_q,
                                           const void* idx_k_pages, float* block_scores,
                                           int32_t* selected, msa_stream_t stream) {
  if (!selected) return MSA_ERR_INVALID_ARG;
  const msa_status st = msa_index_score(cfg, ws, idx_q, idx_k_pages, block_scores, stream);
  return st != MSA_OK ? st : msa_topk_select(cfg, ws, block_scores, selected, stream);
}
