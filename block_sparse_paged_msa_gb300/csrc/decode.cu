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
// consecutive slots of t's selected list.  Design (GB300):
//  * a persistent grid (two 192-thread CTAs per SM) walks the work items
//    (each CTA's first one is its own index, the rest come from a counter);
//    in each CTA a scheduler warp resolves the next items (pages and visible
//    rows of their blocks, the item's Q rows) into a small ring of item
//    records, and a loader warp streams, as soon as a record is out, each
//    selected block's K tile and V tile ([128 tokens][128 dims], contiguous
//    per page and KV head in the HND pool: 32 KiB bf16, 16 KiB e4m3) with 2-D
//    TMA loads (128-byte swizzle) into a ring of shared-memory stages guarded
//    by mbarriers -- so the copies of the next items are already in flight
//    while the current one is being finished;
//  * four consumer warps share every tile: warp w owns tokens [32w, 32w+32),
//    runs S = Q K^T and O += P V on m16n8k16 tensor-core MMAs with the G =
//    H_q / H_kv query heads of the group as the M side (rows >= G are zero),
//    and keeps its own online softmax (exp2 domain); the four states merge once
//    per item and warp 0 writes the normalised partial and its LSE;
//  * rows past the last visible token are masked in S and cleared in V before
//    P V (whatever they hold, 0 * NaN would not vanish): in the V fragments'
//    registers for bf16 tiles, in the converted rows otherwise.  Nothing but
//    the copy engine writes a stage: clearing rows there with ordinary stores
//    gave, now and then, wrong values in another block's V tile of the same
//    CTA, even with a proxy fence before the stage was released;
//  * e4m3 tiles: K feeds an fp16 MMA straight from shared memory (the index
//    dimension is permuted so a thread's four K values of a k-step are one
//    32-bit load), V is converted to fp16 rows by its warp; e4m3 is exact in
//    fp16, k_scale folds into the softmax scale and v_scale into the output;
//  * NVFP4 slots (vLLM MiniMaxM3SparseMSANvfp4Backend: each KV head's keys and
//    values are two slots of packed FP4 data plus block scales) arrive as 1-D
//    bulk copies of 9 KiB per (page, head, K|V) -- 72-byte rows are not a TMA
//    tile shape -- and are dequantised the same way, with another permutation
//    of the head dimension: a thread's eight K values of a pair of k-steps are
//    one 32-bit word of E2M1 codes inside one 16-element scale block, so K =
//    e2m1 x e4m3 is formed in registers (exact in fp16: at most 6 significant
//    bits, magnitudes 2^-10 .. 2688) and V rows likewise.
// msa_combine then merges the splits in a fixed order (deterministic).
#include <cuda.h>

#include <cstring>
#include <mutex>

#include "msa_device.cuh"

namespace msa {
namespace {

constexpr int kConsumers = 4;                      // consumer warps
constexpr int kScheduler = kConsumers;             // warp ids of the two
constexpr int kLoader = kConsumers + 1;            // producer warps
constexpr int kThreads = (kConsumers + 2) * 32;
constexpr int kStages = 3;                         // ring depth (tiles)
constexpr int kTileBytes = kBlock * kHeadDim * 2;  // bf16 tile, 32 KiB
constexpr int kFp8Stages = 4;                      // fp8 tiles are 16 KiB
constexpr int kFp8TileBytes = kBlock * kHeadDim;
constexpr int kFp4Stages = 7;                      // NVFP4 slots are 9 KiB (two CTAs per SM)
constexpr int kFp4TileBytes = kBlock * kFp4Row;

// KV forms of the decode kernel.
enum KvForm { kKvBf16 = 0, kKvFp8 = 1, kKvFp4 = 2 };

template <int KV>
struct KvTraits {
  static constexpr int kStagesN = KV == kKvBf16 ? kStages : (KV == kKvFp8 ? kFp8Stages : kFp4Stages);
  static constexpr int kTile = KV == kKvBf16 ? kTileBytes
                                             : (KV == kKvFp8 ? kFp8TileBytes : kFp4TileBytes);
  static constexpr bool kF16 = KV != kKvBf16;      // fp16 MMAs on dequantised operands
};
constexpr int kConvBytes = 32 * 256;               // per consumer warp: 32 rows, f16
constexpr int kItems = 2;                          // work-item records in flight

// A work item as the producer publishes it: the consumers read only this and
// the item's Q rows (copied next to it), never the global metadata.
struct ItemMeta {
  int t, h, s, nblk;
  int page[32];        // physical page of each usable block, in slot order
  uint8_t ntok[32];    // its visible rows (1..128)
};

struct DecodeArgs {
  int Hkv, Hq, G, S, bps, nsplit, max_blocks, n_items;
  float scale_log2;     // softmax_scale * k_scale * log2(e)
  float v_scale;
  const __nv_bfloat16* q;
  const int32_t* selected;
  const uint8_t* k_pool;   // NVFP4: the pools, read with bulk copies (no tensor map)
  const uint8_t* v_pool;
  // dense paged decode (msa_paged_decode): per (token, KV head) a list of S
  // pages and the number of keys laid out over them; null for the sparse form
  const int32_t* page_table;
  const int32_t* dense_len;
  int num_pages;
};

// The blocks of work item (t, h, split s), as a lane-distributed list: lane i
// (< bps) holds slot s*bps + i; `mask` has a bit for every usable slot (a valid,
// visible block whose page passed the plan's check).  Producer and consumers
// derive it identically.  Sparse form: slot i is selected block j, read through
// the plan's validated block table, with the keys at or before the token's
// position.  Dense form: slot i is page_table[t, h, i], holding keys i*P ..
// of a sequence of dense_len[t, h] keys (pages outside the pool are flagged).
struct ItemBlocks {
  unsigned mask;
  int page, ntok;     // this lane's slot
};

// This lane's raw slot entry, loaded from the item's indices alone (for a
// token of the step, t < num_tokens) so that the load overlaps the token
// metadata reads: sparse form, the selected block; dense form, the page and
// the keys left from the slot on.
struct SlotRaw {
  int v0, v1;
  bool in;            // the lane holds a slot of the item
};

__device__ __forceinline__ SlotRaw slot_raw(const DecodeArgs& a, bool step_token, int t, int h,
                                            int s, int lane) {
  SlotRaw x;
  const int slot0 = s * a.bps;
  x.in = step_token && lane < min(a.bps, a.S - slot0);
  x.v0 = -1;
  x.v1 = 0;
  if (x.in) {
    const int64_t row = (int64_t)t * a.Hkv + h;
    if (a.page_table != nullptr) {
      x.v0 = a.page_table[row * a.S + slot0 + lane];
      x.v1 = a.dense_len[row] - (slot0 + lane) * kBlock;
    } else {
      x.v0 = a.selected[row * a.S + slot0 + lane];
    }
  }
  return x;
}

__device__ __forceinline__ ItemBlocks item_blocks(const WsView& ws, const DecodeArgs& a,
                                                  const SlotRaw& x, int r, int pos, int lane) {
  ItemBlocks b;
  b.page = -1;
  b.ntok = 0;
  bool bad = false;
  if (x.in) {
    if (a.page_table != nullptr) {
      if (x.v1 > 0) {
        if (x.v0 >= 0 && x.v0 < a.num_pages) {
          b.page = x.v0;
          b.ntok = min(kBlock, x.v1);
        } else {
          bad = true;
        }
      }
    } else {
      const int j = x.v0;
      if (j >= 0 && j * kBlock <= pos) {
        b.page = ws.block_table[(int64_t)r * a.max_blocks + j];
        b.ntok = min(kBlock, pos + 1 - j * kBlock);
      }
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(ws.hdr, MSA_DEVERR_PAGE_RANGE);
  b.mask = __ballot_sync(0xffffffffu, b.page >= 0);
  return b;
}

struct Item {
  int t, h, s, r, pos;
  bool active;
};

// Work item idx; num_tokens = the step's tokens (the plan's header, read once).
// The request and the position are independent loads.
__device__ __forceinline__ Item item_of(const WsView& ws, const DecodeArgs& a, int idx,
                                        int num_tokens) {
  Item it;
  it.s = idx % a.nsplit;
  it.h = (idx / a.nsplit) % a.Hkv;
  it.t = idx / (a.nsplit * a.Hkv);
  const bool in = it.t < num_tokens;
  it.r = in ? ws.tok_req[it.t] : -1;
  it.pos = in ? ws.tok_pos[it.t] : -1;
  it.active = it.r >= 0;
  return it;
}

// fp8: the warp converts its 32 rows of an e4m3 V tile (TMA 128-byte swizzle)
// to f16 rows in its private staging area (256-byte swizzled rows), zeroing
// rows past the last visible token.
__device__ __forceinline__ void convert_v_rows(const uint8_t* tile, uint8_t* conv, int warp,
                                               int ntok, int lane) {
  // four inputs at a time ahead of their conversions (the staging stores
  // could alias them for the compiler, which would otherwise chain each load
  // behind the last store)
#pragma unroll
  for (int k0 = 0; k0 < 8; k0 += 4) {
    uint4 win[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int idx = (k0 + k) * 32 + lane;     // 32 rows x 8 chunks of 16 e4m3
      const int row = warp * 32 + (idx >> 3);
      win[k] = row < ntok ? *reinterpret_cast<const uint4*>(tile + swz128(row, idx & 7))
                          : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int idx = (k0 + k) * 32 + lane;
      const int rl = idx >> 3, c = idx & 7;
      const int row = warp * 32 + rl;
      uint32_t o[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      if (row < ntok) {
        const uint4 w = win[k];
        const uint32_t in[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          o[2 * e] = e4m3x2_to_f16x2((uint16_t)(in[e] & 0xffffu));
          o[2 * e + 1] = e4m3x2_to_f16x2((uint16_t)(in[e] >> 16));
        }
      }
      *reinterpret_cast<uint4*>(conv + swz(rl, 2 * c)) = make_uint4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<uint4*>(conv + swz(rl, 2 * c + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
}

// NVFP4: the warp converts its 32 rows of a V slot (72-byte rows: 64 bytes of
// E2M1 codes, 8 E4M3 block scales) to f16 rows in its private staging area
// (256-byte swizzled rows), zeroing rows past the last visible token.
__device__ __forceinline__ void convert_v_rows_fp4(const uint8_t* tile, uint8_t* conv, int warp,
                                                   int ntok, int lane) {
  // four inputs (codes and scale bytes) at a time ahead of their conversions
#pragma unroll
  for (int k0 = 0; k0 < 8; k0 += 4) {
    uint2 win[4];
    uint32_t sin[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int idx = (k0 + k) * 32 + lane;     // 32 rows x 8 blocks of 16 elements
      const int row = warp * 32 + (idx >> 3), c = idx & 7;
      const uint8_t* rp = tile + row * kFp4Row;
      const bool vis = row < ntok;
      win[k] = vis ? *reinterpret_cast<const uint2*>(rp + 8 * c) : make_uint2(0u, 0u);
      sin[k] = vis ? rp[kHeadDim / 2 + c] : 0u;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int idx = (k0 + k) * 32 + lane;
      const int rl = idx >> 3, c = idx & 7;
      const int row = warp * 32 + rl;
      uint32_t o[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      if (row < ntok) {
        const uint2 w = win[k];
        const uint32_t sc = e4m3_scale_f16x2(sin[k]);
        uint32_t lo[4], hi[4];
        e2m1x8_to_f16x2(w.x, lo);
        e2m1x8_to_f16x2(w.y, hi);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          o[e] = hmul2_u32(lo[e], sc);
          o[4 + e] = hmul2_u32(hi[e], sc);
        }
      }
      *reinterpret_cast<uint4*>(conv + swz(rl, 2 * c)) = make_uint4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<uint4*>(conv + swz(rl, 2 * c + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
}

// Persistent split-K decode.  Warp 4 produces: for every block of every work
// item of this CTA it waits for a free ring slot and issues the K and the V
// tile as 2-D TMA loads.  Warps 0-3 consume: warp w owns tokens [32w, 32w+32)
// of every tile, runs S = Q K^T and P V on m16n8k16 tensor-core MMAs with its
// own online softmax, and the four states merge once per work item.
template <int KV>
__global__ void __launch_bounds__(kThreads, 2)
decode_kernel(WsView ws, DecodeArgs a, const __grid_constant__ CUtensorMap tmap_k,
              const __grid_constant__ CUtensorMap tmap_v) {
  constexpr int NST = KvTraits<KV>::kStagesN;
  constexpr int TB = KvTraits<KV>::kTile;
  constexpr bool F16 = KvTraits<KV>::kF16;     // fp16 MMAs, V converted per warp
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem;                                      // NST x TB, 1 KiB aligned
  uint8_t* conv = smem + NST * TB;                           // fp8: 4 x 8 KiB
  uint8_t* qbuf = conv + (F16 ? kConsumers * kConvBytes : 0);   // kItems x G x 256 B
  float* merge = reinterpret_cast<float*>(qbuf + kItems * a.G * 256);
  __shared__ __align__(8) uint64_t full_bar[NST], empty_bar[NST];
  // item_full: a record and its Q rows (consumers); meta_full: the record
  // alone (the loader, which needs only the pages)
  __shared__ __align__(8) uint64_t item_full[kItems], item_empty[kItems], meta_full[kItems];
  __shared__ ItemMeta meta[kItems];
  __shared__ float red_m[kConsumers][16], red_l[kConsumers][16];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kConsumers);
    }
    for (int i = 0; i < kItems; ++i) {
      mbar_init(&item_full[i], 1);
      mbar_init(&meta_full[i], 1);
      mbar_init(&item_empty[i], kConsumers + 1);   // consumers + loader
    }
    fence_barrier_init();
  }
  __syncthreads();
  griddep_launch_dependents();
  griddep_wait();

  if (warp == kScheduler) {
    // -------------------------------------------------------- scheduler
    // Resolves each work item (token metadata and selected slots -> pages) and
    // publishes it with the item's Q rows, up to kItems ahead of the others.
    // After its first item, a CTA takes items from an atomic counter in the
    // workspace header, so CTAs that drew cheap items take more of them.
    int islot = 0;
    uint32_t iphase = 0;
    int nph[kItems] = {0, 0};       // phases armed on item_full[s]
    int qlast[kItems] = {-1, -1};   // phase of the last Q copy on item_full[s]
    // the first item of every CTA is its own index (no counter round trip at
    // the start); the rest come from the counter, after the first gridDim.x
    auto grab = [&]() {
      int i = 0;
      if (lane == 0) i = atomicAdd(&ws.hdr->work_next, 1);
      return (int)gridDim.x + __shfl_sync(0xffffffffu, i, 0);
    };
    const int num_tokens = ws.hdr->num_tokens;
    for (int idx = (int)blockIdx.x; idx < a.n_items; idx = grab()) {
      const int tt = idx / (a.nsplit * a.Hkv);
      const SlotRaw raw = slot_raw(a, tt < num_tokens, tt, (idx / a.nsplit) % a.Hkv,
                                   idx % a.nsplit, lane);
      const Item it = item_of(ws, a, idx, num_tokens);
      if (!it.active) continue;
      const ItemBlocks bl = item_blocks(ws, a, raw, it.r, it.pos, lane);
      if (lane == 0) mbar_wait(&item_empty[islot], iphase ^ 1u, ws.hdr);
      __syncwarp();
      if ((bl.mask >> lane) & 1u) {
        const int p = __popc(bl.mask & ((1u << lane) - 1u));
        meta[islot].ntok[p] = (uint8_t)bl.ntok;
        meta[islot].page[p] = bl.page;
      }
      if (lane == 0) {
        meta[islot].t = it.t;
        meta[islot].h = it.h;
        meta[islot].s = it.s;
        meta[islot].nblk = __popc(bl.mask);
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&meta_full[islot]);              // the loader may start on the pages
        const uint32_t qbytes = (uint32_t)a.G * kHeadDim * 2;
        mbar_arrive_expect_tx(&item_full[islot], qbytes);
        bulk_load(qbuf + islot * qbytes,
                  a.q + ((int64_t)it.t * a.Hq + (int64_t)it.h * a.G) * kHeadDim, qbytes,
                  &item_full[islot]);
        qlast[islot] = nph[islot]++;
      }
      if (++islot == kItems) { islot = 0; iphase ^= 1u; }
    }
    if (lane == 0) {                                      // end-of-work record
      mbar_wait(&item_empty[islot], iphase ^ 1u, ws.hdr);
      meta[islot].t = -1;
      mbar_arrive(&meta_full[islot]);
      mbar_arrive(&item_full[islot]);
      ++nph[islot];
      if (*reinterpret_cast<volatile int*>(&ws.hdr->err) & MSA_DEVERR_TIMEOUT) {
        // a wait gave up: let this warp's Q copies land before the CTA retires
        for (int s2 = 0; s2 < kItems; ++s2)
          if (qlast[s2] >= 0) mbar_drain(&item_full[s2], (uint32_t)(qlast[s2] & 1));
      }
      // the last CTA to stop taking items resets the counters for the next
      // launch on this workspace
      if (atomicAdd(&ws.hdr->work_done, 1) == (int)gridDim.x - 1) {
        ws.hdr->work_next = 0;
        ws.hdr->work_done = 0;
      }
    }
    return;
  }
  if (warp == kLoader) {
    // -------------------------------------------------------------- loader
    // For every published item, the K and V tile of each block as 2-D TMA
    // loads into the stage ring.  Only lane 0 works.
    if (lane == 0) {
      int stage = 0, islot = 0;
      uint32_t phase = 0, iphase = 0;
      int nload = 0;                 // stage arms (one K or V tile each)
      for (;;) {
        mbar_wait(&meta_full[islot], iphase, ws.hdr);
        if (meta[islot].t < 0) break;
        const int nblk = meta[islot].nblk, h = meta[islot].h;
        for (int bi = 0; bi < nblk; ++bi) {
          const int y = (meta[islot].page[bi] * a.Hkv + h) * kBlock;
#pragma unroll
          for (int kind = 0; kind < 2; ++kind) {
            mbar_wait(&empty_bar[stage], phase ^ 1u, ws.hdr);
            mbar_arrive_expect_tx(&full_bar[stage], TB);
            uint8_t* dst = ring + stage * TB;
            if (KV == kKvFp4) {
              // slot 2h (keys) or 2h + 1 (values) of the page
              const int64_t slot = ((int64_t)meta[islot].page[bi] * a.Hkv + h) * 2 + kind;
              bulk_load(dst, (kind == 0 ? a.k_pool : a.v_pool) + slot * TB, TB, &full_bar[stage]);
            } else {
              const void* tm = kind == 0 ? (const void*)&tmap_k : (const void*)&tmap_v;
              tma_load_2d(dst, tm, 0, y, &full_bar[stage]);
              if (KV == kKvBf16) tma_load_2d(dst + TB / 2, tm, 64, y, &full_bar[stage]);
            }
            ++nload;
            if (++stage == NST) { stage = 0; phase ^= 1u; }
          }
        }
        mbar_arrive(&item_empty[islot]);
        if (++islot == kItems) { islot = 0; iphase ^= 1u; }
      }
      // Normally the consumers wait for every tile issued here, so no copy is
      // in flight when the CTA retires.  After a wait gave up they may not
      // have: wait (bounded) for the last phase armed on each stage.
      if (*reinterpret_cast<volatile int*>(&ws.hdr->err) & MSA_DEVERR_TIMEOUT)
        for (int s2 = 0; s2 < NST && s2 < nload; ++s2)
          mbar_drain(&full_bar[s2], (uint32_t)(((nload - 1 - s2) / NST) & 1));
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, tq = lane & 3;
  int stage = 0, islot = 0;
  uint32_t phase = 0, iphase = 0;
  uint8_t* my_conv = conv + warp * kConvBytes;
  for (;;) {
    mbar_wait(&item_full[islot], iphase, ws.hdr);
    const int it_t = meta[islot].t;
    if (it_t < 0) break;                                  // end-of-work record
    const int it_h = meta[islot].h, it_s = meta[islot].s;
    const int nblk = meta[islot].nblk;
    const int my_ntok = lane < nblk ? meta[islot].ntok[lane] : 0;

    // Q fragments from the item's smem copy: rows = the group's query heads
    // (zero past G).  fp8: f16 operands with the index dim permuted so that a
    // thread's four K values of a k-step are one 32-bit shared load
    // (d = 16ks + 4tq + {0,1 | 2,3}).
    uint32_t qa[8][4];
    bool q_ovf = false;             // a query beyond the fp16 range (fp16 operands)
    {
      const __nv_bfloat16* qb =
          reinterpret_cast<const __nv_bfloat16*>(qbuf + islot * a.G * kHeadDim * 2);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int row = g + 8 * hr;
          const __nv_bfloat16* qr = qb + row * kHeadDim;
          if (row >= a.G) {
            qa[ks][hr] = qa[ks][hr + 2] = 0u;
          } else if (KV == kKvFp4) {
            // k-steps 2m, 2m + 1: d = 32 m + 8 tq + 4 (ks & 1) + {0,1 | 2,3}
            const uint2 w =
                *reinterpret_cast<const uint2*>(qr + 32 * (ks >> 1) + 8 * tq + 4 * (ks & 1));
            qa[ks][hr] = bf16x2_to_f16x2(w.x);
            qa[ks][hr + 2] = bf16x2_to_f16x2(w.y);
            q_ovf |= f16x2_has_inf(qa[ks][hr]) | f16x2_has_inf(qa[ks][hr + 2]);
          } else if (F16) {
            const uint2 w = *reinterpret_cast<const uint2*>(qr + ks * 16 + 4 * tq);
            qa[ks][hr] = bf16x2_to_f16x2(w.x);
            qa[ks][hr + 2] = bf16x2_to_f16x2(w.y);
            q_ovf |= f16x2_has_inf(qa[ks][hr]) | f16x2_has_inf(qa[ks][hr + 2]);
          } else {
            qa[ks][hr] = *reinterpret_cast<const uint32_t*>(qr + ks * 16 + 2 * tq);
            qa[ks][hr + 2] = *reinterpret_cast<const uint32_t*>(qr + ks * 16 + 8 + 2 * tq);
          }
        }
      }
    }
    if (F16 && __any_sync(0xffffffffu, q_ovf) && lane == 0) set_error(ws.hdr, MSA_DEVERR_FP16_RANGE);
    __syncwarp();
    if (lane == 0) mbar_arrive(&item_empty[islot]);       // Q and metadata are in registers
    if (++islot == kItems) { islot = 0; iphase ^= 1u; }
    float acc[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY};   // running max (log2 domain), rows g, g+8
    float l_r[2] = {0.f, 0.f};

    for (int bi = 0; bi < nblk; ++bi) {
      const int ntok = __shfl_sync(0xffffffffu, my_ntok, bi);
      // ---------------- K tile: S = Q K^T for this warp's 32 tokens
      mbar_wait(&full_bar[stage], phase, ws.hdr);
      const uint8_t* kt = ring + stage * TB;
      float sc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
        if (KV == kKvFp4) {
          // k-steps 2m, 2m + 1 of this thread: d = 32 m + 8 tq + 0..7, one word
          // of codes inside scale block 2m + tq / 2
          const uint8_t* rp = kt + (warp * 32 + nt * 8 + g) * kFp4Row;
          const uint2 sb = *reinterpret_cast<const uint2*>(rp + kHeadDim / 2);
          const uint32_t s01 = e4m3x2_to_f16x2((uint16_t)(sb.x & 0xffffu));
          const uint32_t s23 = e4m3x2_to_f16x2((uint16_t)(sb.x >> 16));
          const uint32_t s45 = e4m3x2_to_f16x2((uint16_t)(sb.y & 0xffffu));
          const uint32_t s67 = e4m3x2_to_f16x2((uint16_t)(sb.y >> 16));
          const uint32_t sel = (tq >> 1) ? 0x3232u : 0x1010u;   // this thread's half, twice
          const uint32_t spair[4] = {s01, s23, s45, s67};
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(rp + 16 * m + 4 * tq);
            const uint32_t sc2 = __byte_perm(spair[m], 0u, sel);
            uint32_t h[4];
            e2m1x8_to_f16x2(w, h);
            mma_f16(sc[nt], qa[2 * m], hmul2_u32(h[0], sc2), hmul2_u32(h[1], sc2));
            mma_f16(sc[nt], qa[2 * m + 1], hmul2_u32(h[2], sc2), hmul2_u32(h[3], sc2));
          }
        } else if (F16) {
          const int row = warp * 32 + nt * 8 + g;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t w =
                *reinterpret_cast<const uint32_t*>(kt + swz128(row, ks) + 4 * tq);
            mma_f16(sc[nt], qa[ks], e4m3x2_to_f16x2((uint16_t)(w & 0xffffu)),
                    e4m3x2_to_f16x2((uint16_t)(w >> 16)));
          }
        } else {
          const int row = warp * 32 + nt * 8 + (lane & 7);
          const uint32_t kts = smem_u32(kt);
#pragma unroll
          for (int ks = 0; ks < 8; ks += 2) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kts + swz_tma(row, 2 * ks + (lane >> 3)), b0, b1, b2, b3);
            mma_bf16(sc[nt], qa[ks], b0, b1);
            mma_bf16(sc[nt], qa[ks + 1], b2, b3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[stage]);
      if (++stage == NST) { stage = 0; phase ^= 1u; }

      // ---------------- online softmax (log2 domain)
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
      uint32_t pa[2][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const float p0 = exp2f(sc[nt][0] - mref[0]), p1 = exp2f(sc[nt][1] - mref[0]);
        const float p2 = exp2f(sc[nt][2] - mref[1]), p3 = exp2f(sc[nt][3] - mref[1]);
        if (F16) {
          const __half2 h01 = __floats2half2_rn(p0, p1), h23 = __floats2half2_rn(p2, p3);
          const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
          l_r[0] += f01.x + f01.y;
          l_r[1] += f23.x + f23.y;
          pa[nt >> 1][(nt & 1) * 2] = *reinterpret_cast<const uint32_t*>(&h01);
          pa[nt >> 1][(nt & 1) * 2 + 1] = *reinterpret_cast<const uint32_t*>(&h23);
        } else {
          l_r[0] += p0 + p1;
          l_r[1] += p2 + p3;
          pa[nt >> 1][(nt & 1) * 2] = pack_bf16(p0, p1);
          pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p2, p3);
        }
      }

      // ---------------- V tile: O += P V
      mbar_wait(&full_bar[stage], phase, ws.hdr);
      uint8_t* vt = ring + stage * TB;
      uint32_t vbase;
      int vrow0;
      if (F16) {
        if (KV == kKvFp4)
          convert_v_rows_fp4(vt, my_conv, warp, ntok, lane);
        else
          convert_v_rows(vt, my_conv, warp, ntok, lane);
        __syncwarp();
        vbase = smem_u32(my_conv);
        vrow0 = 0;
      } else {
        vbase = smem_u32(vt);
        vrow0 = warp * 32;
      }
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int row = vrow0 + kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
        // bf16: rows past the last visible token may hold anything; P is 0
        // there, but 0 * NaN is not.  The transposed fragments give this
        // thread keys r, r + 1 (b0, b2) and r + 8, r + 9 (b1, b3), r = 16 kk +
        // 2 tq of the warp's 32: mask those halves in registers (the stage
        // itself is written only by the copy engine).
        const int r = warp * 32 + kk * 16 + 2 * tq;
        const uint32_t mlo = (r < ntok ? 0x0000ffffu : 0u) | (r + 1 < ntok ? 0xffff0000u : 0u);
        const uint32_t mhi = (r + 8 < ntok ? 0x0000ffffu : 0u) | (r + 9 < ntok ? 0xffff0000u : 0u);
#pragma unroll
        for (int nd = 0; nd < 16; nd += 2) {
          uint32_t b0, b1, b2, b3;
          if (F16) {
            ldsm_x4_t(vbase + swz(row, nd + (lane >> 4)), b0, b1, b2, b3);
            mma_f16(acc[nd], pa[kk], b0, b1);
            mma_f16(acc[nd + 1], pa[kk], b2, b3);
          } else {
            ldsm_x4_t(vbase + swz_tma(row, nd + (lane >> 4)), b0, b1, b2, b3);
            mma_bf16(acc[nd], pa[kk], b0 & mlo, b1 & mhi);
            mma_bf16(acc[nd + 1], pa[kk], b2 & mlo, b3 & mhi);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[stage]);
      if (++stage == NST) { stage = 0; phase ^= 1u; }
    }

    // ---------------- merge the four warps' states; warp 0 writes the partial
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      l_r[i] += __shfl_xor_sync(0xffffffffu, l_r[i], 1);
      l_r[i] += __shfl_xor_sync(0xffffffffu, l_r[i], 2);
    }
    named_bar_sync(1, kConsumers * 32);            // previous item fully written out
    if (tq == 0) {
      red_m[warp][g] = m_r[0];
      red_m[warp][g + 8] = m_r[1];
      red_l[warp][g] = l_r[0];
      red_l[warp][g + 8] = l_r[1];
    }
    named_bar_sync(1, kConsumers * 32);
    float fw[2], Ltot[2], Mx[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int row = g + 8 * i;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, red_m[w][row]);
      Mx[i] = M;
      fw[i] = M == -INFINITY ? 0.f : exp2f(m_r[i] - M);
      float Ls = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w)
        Ls += M == -INFINITY ? 0.f : red_l[w][row] * exp2f(red_m[w][row] - M);
      Ltot[i] = Ls;
    }
    if (warp > 0) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int row = g + 8 * i;
        if (row >= a.G) continue;
        float* dst = merge + ((warp - 1) * a.G + row) * kHeadDim;
#pragma unroll
        for (int nd = 0; nd < 16; ++nd)
          *reinterpret_cast<float2*>(dst + nd * 8 + 2 * tq) =
              make_float2(acc[nd][2 * i] * fw[i], acc[nd][2 * i + 1] * fw[i]);
      }
    }
    named_bar_sync(1, kConsumers * 32);
    if (warp == 0) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int row = g + 8 * i;
        if (row >= a.G) continue;
        const int64_t hq = (int64_t)it_t * a.Hq + (int64_t)it_h * a.G + row;
        const bool empty = !(Ltot[i] > 0.f);
        const float sc = empty ? 0.f : a.v_scale / Ltot[i];
        float* dst = static_cast<float*>(ws.o_part) + (hq * a.nsplit + it_s) * kHeadDim;
#pragma unroll
        for (int nd = 0; nd < 16; ++nd) {
          float x0 = acc[nd][2 * i] * fw[i], x1 = acc[nd][2 * i + 1] * fw[i];
#pragma unroll
          for (int w = 0; w < kConsumers - 1; ++w) {
            const float2 v = *reinterpret_cast<const float2*>(merge + (w * a.G + row) * kHeadDim +
                                                              nd * 8 + 2 * tq);
            x0 += v.x;
            x1 += v.y;
          }
          *reinterpret_cast<float2*>(dst + nd * 8 + 2 * tq) = make_float2(x0 * sc, x1 * sc);
        }
        if (tq == 0)
          ws.lse_part[hq * a.nsplit + it_s] = empty ? -INFINITY : (Mx[i] + log2f(Ltot[i])) * kLn2;
      }
    }
  }
}

// ---- combine (decode): one warp per (token, query head), splits merged in a
// fixed order.
__global__ void __launch_bounds__(256)
combine_kernel(WsView ws, int Hq, int nsplit, __nv_bfloat16* __restrict__ out,
               float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int64_t idx = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int t = (int)(idx / Hq);
  griddep_launch_dependents();
  griddep_wait();
  if (t >= ws.hdr->num_tokens) return;
  const bool active = ws.tok_req[t] >= 0;
  const float* lp = ws.lse_part + idx * nsplit;
  float M = -INFINITY;
  if (active)
    for (int s = lane; s < nsplit; s += 32) M = fmaxf(M, lp[s]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    float L = 0.f;
    for (int s = 0; s < nsplit; ++s) L += exp2f((lp[s] - M) * kLog2e);
    const float lse_tot = M + logf(L);
    for (int s = 0; s < nsplit; ++s) {
      const float w = expf(lp[s] - lse_tot);
      const float4 v = *reinterpret_cast<const float4*>(static_cast<const float*>(ws.o_part) +
                                                        (idx * nsplit + s) * kHeadDim + 4 * lane);
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

// ---- combine (prefill): 16 threads per (token, query head), 8 dimensions
// each.  The token's selected blocks are its slots 0 .. min(nb, S) - 1 (nb =
// its visible blocks); slot s of (t, KV head h) is CSR entry slot_entry[t, h,
// s], whose fp16 partial row is entry * G + g.  Thread c of the group looks up
// the entries and LSEs of slots c and 16 + c (slots from 32 on are looked up
// again in each pass) and the group shares them by shuffles, so that the
// partial rows load independently of one another.  Merged in slot order.
__device__ __forceinline__ void combine_rows(const uint4* __restrict__ part, int64_t row, float w,
                                             int n, int c, unsigned gmask, float (&o)[8]) {
#pragma unroll
  for (int k0 = 0; k0 < 16; k0 += 8) {
    if (k0 >= n) break;                          // uniform per group
    uint4 raw[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int64_t rk = __shfl_sync(gmask, row, k0 + k, 16);
      raw[k] = k0 + k < n ? __ldg(part + rk * (kHeadDim / 8) + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float wk = __shfl_sync(gmask, w, k0 + k, 16);
      const uint32_t u[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[q]));
        o[2 * q] = fmaf(wk, f.x, o[2 * q]);
        o[2 * q + 1] = fmaf(wk, f.y, o[2 * q + 1]);
      }
    }
  }
}

__global__ void __launch_bounds__(256, 4)
combine_prefill_kernel(WsView ws, int Hq, int Hkv, int S, __nv_bfloat16* __restrict__ out,
                       float* __restrict__ lse) {
  const int64_t idx = (int64_t)blockIdx.x * 16 + (threadIdx.x >> 4);
  const int c = threadIdx.x & 15;
  const unsigned gmask = 0xffffu << (threadIdx.x & 16);   // this half-warp
  griddep_launch_dependents();
  griddep_wait();
  const int t = (int)(idx / Hq);
  if (t >= ws.hdr->num_tokens) return;                    // uniform per half-warp
  const int hq = (int)(idx % Hq), G = Hq / Hkv, h = hq / G, g = hq % G;
  const int nvalid = ws.tok_req[t] >= 0 ? min(S, ws.tok_pos[t] / kBlock + 1) : 0;
  const int32_t* ent = ws.slot_entry + ((int64_t)t * Hkv + h) * S;
  auto lookup = [&](int s, int64_t& row, float& x) {
    row = 0;
    x = -INFINITY;
    if (s < nvalid) {
      row = (int64_t)__ldg(ent + s) * G + g;
      x = __ldg(ws.lse_part + row);
    }
  };
  int64_t r0, r1;
  float x0, x1;
  lookup(c, r0, x0);
  lookup(16 + c, r1, x1);
  // max and sum of exp over the slots' LSE
  float M = fmaxf(x0, x1);
  for (int s0 = 32; s0 < nvalid; s0 += 16) {
    int64_t rr;
    float xx;
    lookup(s0 + c, rr, xx);
    M = fmaxf(M, xx);
  }
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(gmask, M, o, 16));
  float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float lse_tot = -INFINITY;
  if (M != -INFINITY) {
    float L = exp2f((x0 - M) * kLog2e) + exp2f((x1 - M) * kLog2e);
    for (int s0 = 32; s0 < nvalid; s0 += 16) {
      int64_t rr;
      float xx;
      lookup(s0 + c, rr, xx);
      L += exp2f((xx - M) * kLog2e);
    }
#pragma unroll
    for (int o2 = 8; o2 >= 1; o2 >>= 1) L += __shfl_xor_sync(gmask, L, o2, 16);
    lse_tot = M + logf(L);
    const uint4* part = static_cast<const uint4*>(ws.o_part);
    combine_rows(part, r0, expf(x0 - lse_tot), min(16, nvalid), c, gmask, o);
    if (nvalid > 16) combine_rows(part, r1, expf(x1 - lse_tot), min(16, nvalid - 16), c, gmask, o);
    for (int s0 = 32; s0 < nvalid; s0 += 16) {
      int64_t rr;
      float xx;
      lookup(s0 + c, rr, xx);
      combine_rows(part, rr, expf(xx - lse_tot), min(16, nvalid - s0), c, gmask, o);
    }
  }
  if (c == 0) lse[idx] = lse_tot;
  uint32_t pk[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    __nv_bfloat162 b = __floats2bfloat162_rn(o[2 * k], o[2 * k + 1]);
    pk[k] = *reinterpret_cast<uint32_t*>(&b);
  }
  reinterpret_cast<uint4*>(out + idx * kHeadDim)[c] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
}

template <int KV>
size_t decode_smem(int G) {
  const size_t ring = (size_t)KvTraits<KV>::kStagesN * KvTraits<KV>::kTile;
  const size_t conv = KvTraits<KV>::kF16 ? (size_t)kConsumers * kConvBytes : 0;
  return ring + conv + (size_t)kItems * G * kHeadDim * 2 +
         (size_t)(kConsumers - 1) * G * kHeadDim * 4;
}

template <int KV>
msa_status launch_decode(const WsView& v, const DecodeArgs& a, const CUtensorMap& tk,
                         const CUtensorMap& tv, cudaStream_t s) {
  static std::mutex mu;
  static int grid_per_dev[64] = {0};
  static size_t smem_set[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return MSA_ERR_CUDA;
  const size_t smem = decode_smem<KV>(a.G);
  int grid;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (smem_set[dev] < smem) {
      if (cudaFuncSetAttribute(decode_kernel<KV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem) != cudaSuccess)
        return MSA_ERR_CUDA;
      smem_set[dev] = smem;
      grid_per_dev[dev] = 0;
    }
    if (grid_per_dev[dev] == 0) {
      int per_sm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<KV>, kThreads,
                                                        smem) != cudaSuccess)
        return MSA_ERR_CUDA;
      grid_per_dev[dev] = sm_count() * (per_sm > 0 ? per_sm : 1);
    }
    grid = grid_per_dev[dev];
  }
  if (grid > a.n_items) grid = a.n_items;
  if (grid <= 0) return MSA_OK;
  return launch_pdl(decode_kernel<KV>, dim3(grid), dim3(kThreads), smem, s, v, a, tk, tv);
}

}  // namespace
}  // namespace msa

using namespace msa;

namespace msa {
namespace {
// The decode pipeline for either form: `selected` (sparse) or `page_table` +
// `dense_len` (dense paged decode over compacted pages).
msa_status decode_common(const msa_config* cfg, void* ws, const void* q, const void* k_pages,
                         const void* v_pages, const int32_t* selected,
                         const int32_t* page_table, const int32_t* dense_len,
                         cudaStream_t s) {
  msa_status st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (is_prefill(*cfg)) return MSA_ERR_INVALID_ARG;   // prefill uses msa_sparse_prefill
  if (!ws || !q || !k_pages || !v_pages || (!selected && !(page_table && dense_len)))
    return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages)) return MSA_ERR_INVALID_ARG;
  DecodeArgs a;
  a.Hkv = cfg->num_kv_heads;
  a.Hq = cfg->num_q_heads;
  a.G = cfg->num_q_heads / cfg->num_kv_heads;
  a.S = width_of(*cfg);
  a.bps = blocks_per_split_of(*cfg);
  if (a.bps > 32) return MSA_ERR_UNSUPPORTED;   // one warp lists a split's blocks
  a.nsplit = splits_of(*cfg);
  a.max_blocks = cfg->max_blocks_per_req;
  const int64_t items = (int64_t)max_tokens_of(*cfg) * a.Hkv * a.nsplit;
  if (items <= 0) return MSA_OK;
  if (items > 0x7fffffff) return MSA_ERR_UNSUPPORTED;
  a.n_items = (int)items;
  const bool scaled = cfg->kv_dtype != MSA_KV_BF16;
  a.scale_log2 = cfg->softmax_scale * (scaled ? cfg->k_scale : 1.f) * kLog2e;
  a.v_scale = scaled ? cfg->v_scale : 1.f;
  a.q = (const __nv_bfloat16*)q;
  a.selected = selected;
  a.k_pool = (const uint8_t*)k_pages;
  a.v_pool = (const uint8_t*)v_pages;
  a.page_table = page_table;
  a.dense_len = dense_len;
  a.num_pages = cfg->num_pages;
  const WsView v = view_of(*cfg, ws);
  CUtensorMap tk, tv;
  if (cfg->kv_dtype == MSA_KV_NVFP4) {
    memset(&tk, 0, sizeof(tk));      // bulk copies from the pool pointers instead
    memset(&tv, 0, sizeof(tv));
    return launch_decode<kKvFp4>(v, a, tk, tv, s);
  }
  const bool fp8 = cfg->kv_dtype == MSA_KV_FP8_E4M3;
  const int64_t rows = (int64_t)cfg->num_pages * a.Hkv * kBlock;
  if (rows > 0x7fffffff) return MSA_ERR_UNSUPPORTED;   // TMA row coordinates are int32
  if (!make_pool_map(&tk, k_pages, rows, fp8) || !make_pool_map(&tv, v_pages, rows, fp8))
    return MSA_ERR_CUDA;
  return fp8 ? launch_decode<kKvFp8>(v, a, tk, tv, s) : launch_decode<kKvBf16>(v, a, tk, tv, s);
}
}  // namespace
}  // namespace msa

extern "C" msa_status msa_sparse_decode(const msa_config* cfg, void* ws, const void* q,
                                        const void* k_pages, const void* v_pages,
                                        const int32_t* selected, msa_stream_t stream) {
  if (selected == nullptr) return MSA_ERR_INVALID_ARG;
  return decode_common(cfg, ws, q, k_pages, v_pages, selected, nullptr, nullptr,
                       (cudaStream_t)stream);
}

extern "C" msa_status msa_paged_decode(const msa_config* cfg, void* ws, const void* q,
                                       const void* k_pages, const void* v_pages,
                                       const int32_t* page_table, const int32_t* seq_lens,
                                       msa_stream_t stream) {
  if (page_table == nullptr || seq_lens == nullptr) return MSA_ERR_INVALID_ARG;
  return decode_common(cfg, ws, q, k_pages, v_pages, nullptr, page_table, seq_lens,
                       (cudaStream_t)stream);
}

namespace msa {
namespace {
// One CTA waits on an mbarrier that no thread ever arrives on, with a short
// poll limit: the bounded wait must give up, record MSA_DEVERR_TIMEOUT and
// return, leaving the context usable.
__global__ void __launch_bounds__(32) selftest_wait_kernel(WsView ws) {
  __shared__ __align__(8) uint64_t never;
  if (threadIdx.x == 0) {
    mbar_init(&never, 1);
    fence_barrier_init();
  }
  __syncwarp();
  griddep_launch_dependents();
  griddep_wait();
  mbar_wait<1u << 14>(&never, 0, ws.hdr);
}
}  // namespace
}  // namespace msa

extern "C" msa_status msa_selftest_wait_timeout(const msa_config* cfg, void* ws,
                                                msa_stream_t stream) {
  msa_status st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (!ws) return MSA_ERR_INVALID_ARG;
  return launch_pdl(selftest_wait_kernel, dim3(1), dim3(32), 0, (cudaStream_t)stream,
                    view_of(*cfg, ws));
}

extern "C" msa_status msa_combine(const msa_config* cfg, const void* ws, void* out, float* lse,
                                  msa_stream_t stream) {
  msa_status st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (!ws || !out || !lse) return MSA_ERR_INVALID_ARG;
  if (((uintptr_t)out & (is_prefill(*cfg) ? 15 : 7)) != 0) return MSA_ERR_INVALID_ARG;
  const int64_t items = (int64_t)max_tokens_of(*cfg) * cfg->num_q_heads;
  if (items <= 0) return MSA_OK;
  const WsView v = view_of(*cfg, ws);
  if (is_prefill(*cfg)) {
    const int64_t pgrid = (items + 15) / 16;
    if (pgrid > 0x7fffffff) return MSA_ERR_UNSUPPORTED;
    return launch_pdl(combine_prefill_kernel, dim3((unsigned)pgrid), dim3(256), 0,
                      (cudaStream_t)stream, v, cfg->num_q_heads, cfg->num_kv_heads,
                      width_of(*cfg), (__nv_bfloat16*)out, lse);
  }
  const int64_t grid = (items + 7) / 8;
  if (grid > 0x7fffffff) return MSA_ERR_UNSUPPORTED;
  return launch_pdl(combine_kernel, dim3((unsigned)grid), dim3(256), 0,
                    (cudaStream_t)stream, v, cfg->num_q_heads, splits_of(*cfg),
                    (__nv_bfloat16*)out, lse);
}
