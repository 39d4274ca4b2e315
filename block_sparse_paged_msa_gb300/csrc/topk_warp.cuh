// The warp-wide top-k selection of one (token, KV head) row: msa_topk_select
// (topk.cu) runs it for rows of up to 1 024 candidates.  Not part of the ABI.
#pragma once

#include "msa_internal.cuh"

namespace msa {

__device__ __forceinline__ uint32_t topk_order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One warp, one (token, KV head) row, for up to 32 * CPL candidates, kept in registers
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
__device__ __forceinline__ void topk_row(const WsView& ws, int64_t row, int Hkv, int max_blocks,
                                         int init, int local, int topk, int S,
                                         const float* __restrict__ scores,
                                         int* __restrict__ selected, int* hist, int lane) {
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
    key[i] = c < nc ? topk_order_key(__ldcg(sc + c0 + c)) : 0u;
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


}  // namespace msa
