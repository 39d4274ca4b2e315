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
#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kThreads = 128;

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

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
  for (int i = tid; i < nc; i += kThreads) keys[i] = order_key(sc[c0 + i]);
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

// Warp per (token, KV head) for up to 32 * CPL candidates, kept in registers
// (lane l holds candidates l, l + 32, ...).  The key of the k-th best
// candidate is found 8 bits at a time from the top (an MSB-first radix
// select): per pass the warp builds a 256-bin histogram of the candidates
// that match the digits fixed so far (shared-memory atomics, one histogram
// per warp), a descending scan over the bins finds the bin holding the k-th
// best, and its count above that bin is taken.  The output is the init
// blocks, then the winning candidates in ascending order (ties among equal
// keys by lower index), then the local blocks -- already ascending, since
// init < candidates < local.
template <int CPL>
__global__ void __launch_bounds__(256)
topk_warp_kernel(WsView ws, int Hkv, int max_blocks, int init, int local, int topk, int S,
                 const float* __restrict__ scores, int* __restrict__ selected) {
  __shared__ int whist[8][256];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int* hist = whist[wid];
  const int64_t row = (int64_t)blockIdx.x * 8 + wid;                  // (token, KV head)
  griddep_launch_dependents();
  griddep_wait();
  if (row >= (int64_t)ws.hdr->num_tokens * Hkv) return;               // warp-uniform
  const int t = (int)(row / Hkv);
  int* out = selected + row * S;
  if (ws.tok_req[t] < 0) {
    for (int i = lane; i < S; i += 32) out[i] = -1;
    return;
  }
  const int nb = ws.tok_pos[t] / kBlock + 1;
  const float* sc = scores + row * max_blocks;
  const int c0 = min(init, nb);
  const int c1 = max(c0, nb - local);   // candidates are [c0, c1)
  const int nc = c1 - c0;
  const int K = min(topk, nc);
  uint32_t key[CPL];
  uint32_t kmax = 0u;                           // over this lane's candidates
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = i * 32 + lane;
    key[i] = c < nc ? order_key(sc[c0 + c]) : 0u;
    kmax = max(kmax, key[i]);
  }
  uint32_t thr = 0xffffffffu;   // keys > thr win outright
  int ktie = 0;                 // this many keys == thr win, lowest index first
  if (K == nc) {
    thr = 0u;                   // every candidate (real keys are >= 1)
  } else if (K > 0) {
    // Only the bytes where the candidates' keys differ need a pass: diff = the
    // OR over candidates of (key ^ largest key).  Above its highest byte every
    // key matches the largest one, below its lowest every key carries the same
    // bits (integer-valued scores share their top byte and their low mantissa
    // bytes, so one pass is typical).
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    uint32_t dl = 0u;
#pragma unroll
    for (int i = 0; i < CPL; ++i)
      if (i * 32 + lane < nc) dl |= key[i] ^ kmax;
    const uint32_t diff = __reduce_or_sync(0xffffffffu, dl);
    // all keys equal: the K lowest indices win (diff = 0 -> no pass)
    const int top = diff ? (31 - __clz(diff)) >> 3 << 3 : -8;   // first shift
    const int bot = diff ? (__ffs(diff) - 1) >> 3 << 3 : 0;     // last shift
    uint32_t mask = top >= 24 ? 0u : 0xffffffffu << (top + 8);
    uint32_t prefix = kmax & mask;
    int krem = K;
#pragma unroll 1
    for (int shift = top; shift >= bot; shift -= 8) {
#pragma unroll
      for (int e = 0; e < 8; ++e) hist[lane * 8 + e] = 0;
      __syncwarp();
#pragma unroll
      for (int i = 0; i < CPL; ++i)
        if (i * 32 + lane < nc && (key[i] & mask) == prefix)
          atomicAdd(&hist[(key[i] >> shift) & 255], 1);
      __syncwarp();
      // lane l owns bins 255 - 8l .. 248 - 8l (descending)
      int cnt[8], tot = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        cnt[e] = hist[255 - 8 * lane - e];
        tot += cnt[e];
      }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, incl >= krem);
      const int L = __ffs(hit) - 1;          // lane whose bins hold the k-th best
      int bin = 0, rem = 0;
      if (lane == L) {
        int c = incl - tot;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (c + cnt[e] >= krem) {
            bin = 255 - 8 * lane - e;
            rem = krem - c;
            break;
          }
          c += cnt[e];
        }
      }
      bin = __shfl_sync(0xffffffffu, bin, L);
      krem = __shfl_sync(0xffffffffu, rem, L);
      prefix |= (uint32_t)bin << shift;
      mask |= 0xffu << shift;
      __syncwarp();
    }
    thr = prefix | (kmax & ~mask);   // the bits below the last pass are shared
    ktie = krem;
  }
  for (int i = lane; i < c0; i += 32) out[i] = i;
  int tie_carry = 0, sel_carry = 0;
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    if (i * 32 >= nc) break;                                          // warp-uniform
    const int c = i * 32 + lane;
    const bool cand = c < nc;
    const bool tie = cand && key[i] == thr;
    const unsigned tb = __ballot_sync(0xffffffffu, tie);
    const int tie_rank = tie_carry + __popc(tb & ((1u << lane) - 1u));
    const bool sel = cand && (key[i] > thr || (tie && tie_rank < ktie));
    const unsigned sb = __ballot_sync(0xffffffffu, sel);
    if (sel) out[c0 + sel_carry + __popc(sb & ((1u << lane) - 1u))] = c0 + c;
    tie_carry += __popc(tb);
    sel_carry += __popc(sb);
  }
  const int nl = nb - c1;
  for (int i = lane; i < nl; i += 32) out[c0 + sel_carry + i] = c1 + i;
  for (int i = c0 + sel_carry + nl + lane; i < S; i += 32) out[i] = -1;
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
