// msa_topk_select: init blocks U local blocks U the top-k remaining blocks by
// (score descending, block index ascending), written ascending and -1 padded.
//
// sglang MiniMaxSparseAttnBackend.__init__ resolves init_blocks, local_blocks
// (= ceil(local_tokens / block) + 1) and topk_blocks; vLLM
// MiniMaxM3SparseMSAImpl.forward consumes the resulting per-token, per-KV-head
// selected-block lists ([tokens, H, MK]).  The tie rule (lower index wins) is
// this library's specification; the pages leave it open.
//
// Design: one 128-thread CTA per (token, KV head).  The candidate scores are
// mapped to order-preserving 32-bit keys in shared memory; an MSB-first radix
// select (4 passes of 8 bits, shared-memory histograms, a warp scan over the
// 256 bins) finds the exact key of the k-th best candidate and how many of the
// candidates equal to it are taken; one ordered pass then marks the winners
// (ties by ascending index, via ballot prefix counts) and compacts the
// selected block ids in ascending order.  Deterministic, no sort needed.
#include "topk_warp.cuh"

namespace msa {
namespace {

constexpr int kThreads = 128;

// Exclusive prefix count of `flag` over the CTA in thread order, and the total.
__device__ __forceinline__ int cta_prefix(bool flag, int* warp_cnt, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  if (lane == 0) warp_cnt[warp] = __popc(bal);
  __syncthreads();
  int before = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const int c = warp_cnt[w];
    if (w < warp) before += c;
    total += c;
  }
  __syncthreads();
  return before + __popc(bal & ((1u << lane) - 1u));
}

__global__ void __launch_bounds__(kThreads)
topk_kernel(WsView ws, int Hkv, int max_blocks, int init, int local, int topk, int S,
            const float* __restrict__ scores, int* __restrict__ selected) {
  extern __shared__ uint32_t keys[];  // [max_blocks]
  __shared__ int hist[256];
  __shared__ int warp_cnt[kThreads / 32];
  __shared__ int pick_bin, pick_rem;
  const int tid = threadIdx.x;
  const int t = blockIdx.x / Hkv, h = blockIdx.x % Hkv;
  griddep_launch_dependents();
  griddep_wait();
  if (t >= ws.hdr->num_tokens) return;
  int* out = selected + ((int64_t)t * Hkv + h) * S;
  const int r = ws.tok_req[t];
  if (r < 0) {
    for (int i = tid; i < S; i += kThreads) out[i] = -1;
    return;
  }
  const int nb = ws.tok_pos[t] / kBlock + 1;
  const float* sc = scores + ((int64_t)t * Hkv + h) * max_blocks;
  const int c0 = min(init, nb);
  const int c1 = max(c0, nb - local);   // candidates are [c0, c1)
  const int nc = c1 - c0;
  const int K = min(topk, nc);
  for (int i = tid; i < nc; i += kThreads) keys[i] = topk_order_key(sc[c0 + i]);
  __syncthreads();

  uint32_t thr = 0xffffffffu;  // keys > thr win outright
  int ktie = 0;                // this many keys == thr win, lowest index first
  if (K == nc) {
    thr = 0;
    ktie = nc;                 // every candidate is taken (keys >= 0)
  } else if (K > 0) {
    uint32_t prefix = 0, mask = 0;
    int krem = K;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int b = tid; b < 256; b += kThreads) hist[b] = 0;
      __syncthreads();
      for (int i = tid; i < nc; i += kThreads) {
        const uint32_t k = keys[i];
        if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255], 1);
      }
      __syncthreads();
      if (tid < 32) {
        // lane l owns bins 255-8l .. 248-8l (descending)
        int cnt = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) cnt += hist[255 - 8 * tid - e];
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (tid >= o) incl += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, incl >= krem);
        const int L = __ffs(hit) - 1;
        if (tid == L) {
          int c = incl - cnt;
          for (int e = 0; e < 8; ++e) {
            const int bin = 255 - 8 * tid - e;
            if (c + hist[bin] >= krem) {
              pick_bin = bin;
              pick_rem = krem - c;
              break;
            }
            c += hist[bin];
          }
        }
      }
      __syncthreads();
      prefix |= (uint32_t)pick_bin << shift;
      mask |= 0xffu << shift;
      krem = pick_rem;
      __syncthreads();
    }
    thr = prefix;
    ktie = krem;
  }

  // Ordered pass over j in [0, nb): mark and compact.
  int tie_carry = 0, sel_carry = 0;
  for (int base = 0; base < nb; base += kThreads) {
    const int j = base + tid;
    const bool in = j < nb;
    const bool cand = in && j >= c0 && j < c1;
    const uint32_t k = cand ? keys[j - c0] : 0u;
    const bool tie = cand && k == thr;
    int tie_total;
    const int tie_rank = tie_carry + cta_prefix(tie, warp_cnt, tie_total);
    const bool sel = in && (!cand || k > thr || (tie && tie_rank < ktie));
    int sel_total;
    const int pos = sel_carry + cta_prefix(sel, warp_cnt, sel_total);
    if (sel) out[pos] = j;
    tie_carry += tie_total;
    sel_carry += sel_total;
  }
  for (int i = sel_carry + tid; i < S; i += kThreads) out[i] = -1;
}

// Warp per (token, KV head) for up to 32 * CPL candidates (topk_warp.cuh).
template <int CPL>
__global__ void __launch_bounds__(256)
topk_warp_kernel(WsView ws, int Hkv, int max_blocks, int init, int local, int topk, int S,
                 const float* __restrict__ scores, int* __restrict__ selected) {
  __shared__ int whist[8][256];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t row = (int64_t)blockIdx.x * 8 + wid;                  // (token, KV head)
  griddep_launch_dependents();
  griddep_wait();
  if (row >= (int64_t)ws.hdr->num_tokens * Hkv) return;               // warp-uniform
  topk_row<CPL>(ws, row, Hkv, max_blocks, init, local, topk, S, scores, selected, whist[wid],
                lane);
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" msa_status msa_topk_select(const msa_config* cfg, const void* ws,
                                      const float* block_scores, int32_t* selected,
                                      msa_stream_t stream) {
  msa_status st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (!ws || !block_scores || !selected) return MSA_ERR_INVALID_ARG;
  const WsView v = view_of(*cfg, ws);
  const int64_t grid = (int64_t)max_tokens_of(*cfg) * cfg->num_kv_heads;
  if (grid <= 0) return MSA_OK;
  if (grid > 0x7fffffff) return MSA_ERR_UNSUPPORTED;
  // up to 1 024 candidates: a warp per (token, KV head), candidates in registers
  const int nbmax = cfg->max_blocks_per_req;
  if (nbmax <= 1024) {
    const int64_t wgrid = (grid + 7) / 8;
    auto kern = nbmax <= 256 ? topk_warp_kernel<8> : topk_warp_kernel<32>;
    return launch_pdl(kern, dim3((unsigned)wgrid), dim3(256), 0, (cudaStream_t)stream, v,
                      cfg->num_kv_heads, nbmax, cfg->init_blocks, cfg->local_blocks,
                      cfg->topk_blocks, width_of(*cfg), block_scores, selected);
  }
  const size_t smem = sizeof(uint32_t) * cfg->max_blocks_per_req;
  return launch_pdl(topk_kernel, dim3((unsigned)grid), dim3(kThreads), smem,
                    (cudaStream_t)stream, v, cfg->num_kv_heads, cfg->max_blocks_per_req,
                    cfg->init_blocks, cfg->local_blocks, cfg->topk_blocks, width_of(*cfg),
                    block_scores, selected);
}
