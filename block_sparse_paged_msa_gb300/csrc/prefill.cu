// Chunked-prefill path: the key-block -> query CSR and block-sparse attention
// tiles per CSR row (the chunk's index scores are in prefill_index.cu).
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
//  * csr_mark / csr_count / csr_fill kernels: the CSR built token-major from
//    per-(KV head, key block) token bitmaps, so every row lists its tokens
//    ascending and the structure is deterministic.
//  * prefill_tc_kernel (msa_sparse_prefill): fifth-generation tensor cores.
//    A persistent CTA per SM walks work items of up to 32 M-tiles of one CSR
//    row; per row the K and V tiles arrive by TMA and V is converted to fp16
//    in place (read by P V as an MN-major operand).  M-tiles of 128 rows
//    (tokens x GQA heads) alternate between two softmax warpgroups: one
//    thread issues tcgen05.mma for S = Q K^T (bf16) and O = P V (fp16, P from
//    TMEM) with fp32 accumulators in TMEM; each warpgroup thread owns one row
//    (tcgen05.ld), applies the causal mask and the softmax; the normalised
//    fp16 partial rows of a tile, contiguous in CSR-entry order, leave by TMA
//    tile stores with their LSE beside them.  msa_combine merges each token's
//    slots.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "tcgen05.cuh"

namespace msa {
namespace {

// ------------------------------------------------------------ CSR
// Row (h, r, j) of the key-block -> query CSR lists, ascending, the tokens of
// request r whose selection for KV head h holds block j.  Built token-major
// and deterministically: every selected entry sets its token's bit in the
// bitmap of (h, j) (csr_mark_kernel); a warp per row counts the bits of the
// request's words and records the count before each word (csr_count_kernel);
// after the scan of the counts, an entry's CSR position is the row start +
// the bits before it (csr_fill_kernel).  An entry counts when its block is
// visible to the token (j <= position / P, j < the request's block count).

struct CsrEntry {
  bool ok;
  int r, j;
  int64_t word;      // bitmap word of (h, j, token)
  uint32_t bit;
};

__device__ __forceinline__ CsrEntry csr_entry(const WsView& ws, const int32_t* selected, int t,
                                              int h, int s, int Hkv, int NB, int S,
                                              int64_t wpr) {
  CsrEntry c;
  c.ok = false;
  c.r = ws.tok_req[t];
  if (c.r < 0) return c;
  c.j = selected[((int64_t)t * Hkv + h) * S + s];
  if (c.j < 0 || c.j >= NB || c.j >= ws.req_nb[c.r] || c.j * kBlock > ws.tok_pos[t]) return c;
  const int qs = ws.req_qstart[c.r];
  const int wl = t - qs;
  c.word = ((int64_t)h * NB + c.j) * wpr + (qs >> 5) + c.r + (wl >> 5);
  c.bit = 1u << (wl & 31);
  c.ok = true;
  return c;
}

__global__ void __launch_bounds__(256)
csr_mark_kernel(WsView ws, int Hkv, int NB, int S, int64_t wpr, const int32_t* __restrict__ selected) {
  griddep_launch_dependents();
  griddep_wait();
  const int64_t n = (int64_t)ws.hdr->num_tokens * Hkv * S;
  for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256) {
    const int s = (int)(i % S), h = (int)((i / S) % Hkv), t = (int)(i / ((int64_t)S * Hkv));
    const CsrEntry c = csr_entry(ws, selected, t, h, s, Hkv, NB, S, wpr);
    if (c.ok) atomicOr(ws.csr_bits + c.word, c.bit);
  }
}

// One warp per row (h, r, j): popcounts of request r's words, exclusive
// prefix per word, the row's count into row_ptr[row + 1].
__global__ void __launch_bounds__(256)
csr_count_kernel(WsView ws, int Hkv, int B, int NB, int64_t wpr, int32_t* __restrict__ row_ptr) {
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  griddep_launch_dependents();
  griddep_wait();
  if (row >= (int64_t)Hkv * B * NB) return;
  const int j = (int)(row % NB);
  const int r = (int)((row / NB) % B);
  const int h = (int)(row / ((int64_t)NB * B));
  int total = 0;
  if (r < ws.hdr->batch && j < ws.req_nb[r]) {
    const int qs = ws.req_qstart[r], nq = ws.req_qstart[r + 1] - qs;
    const int64_t base = ((int64_t)h * NB + j) * wpr + (qs >> 5) + r;
    const int nw = (nq + 31) >> 5;
    for (int w0 = 0; w0 < nw; w0 += 32) {
      const int w = w0 + lane;
      const int c = w < nw ? __popc(ws.csr_bits[base + w]) : 0;
      int x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (w < nw) ws.csr_wpre[base + w] = total + x - c;
      total += __shfl_sync(0xffffffffu, x, 31);
    }
  }
  if (lane == 0) {
    row_ptr[row + 1] = total;
    if (row == 0) row_ptr[0] = 0;
  }
}

__global__ void __launch_bounds__(256)
csr_fill_kernel(WsView ws, int Hkv, int B, int NB, int S, int64_t wpr,
                const int32_t* __restrict__ selected, const int32_t* __restrict__ row_ptr,
                int32_t* __restrict__ q_idx) {
  griddep_launch_dependents();
  griddep_wait();
  const int64_t n = (int64_t)ws.hdr->num_tokens * Hkv * S;
  for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256) {
    const int s = (int)(i % S), h = (int)((i / S) % Hkv), t = (int)(i / ((int64_t)S * Hkv));
    const CsrEntry c = csr_entry(ws, selected, t, h, s, Hkv, NB, S, wpr);
    if (!c.ok) continue;
    const int64_t row = ((int64_t)h * B + c.r) * NB + c.j;
    const int e = row_ptr[row] + ws.csr_wpre[c.word] + __popc(ws.csr_bits[c.word] & (c.bit - 1u));
    q_idx[e] = t;
    ws.slot_entry[i] = e;
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
// Work items: a CSR row's tokens in chunks of kTilesPerItem M-tiles of 128
// rows (tokens x GQA heads); msa_build_k2q_csr writes the first item of every
// row (ws.sched) and the items ordered largest first (ws.item_order: CSR row,
// first and end entry of each), so the huge rows of the init / local blocks
// are split and the CTAs' round-robin shares come out even.  The item size
// sets how evenly the round-robin lands: over the sorted items of the
// 4 x (16 384 + 2 048)-token prefill, the busiest CTA's share of tiles is 1.09
// x the mean with items of 32 M-tiles and 1.02 x with 20 (simulated from the
// step's CSR; measured 0.932 -> 0.889 ms per launch with the issue order below).
constexpr int kTilesPerItem = 20;
// the workspace bounds the items by one per 128 CSR entries per row (an item
// holds kTilesPerItem * 128 / G >= 8 kTilesPerItem tokens, G <= 16)
static_assert(kTilesPerItem * 8 >= 128, "item bound of the workspace layout");
constexpr int kLoaderWarps = 3;          // Q loaders (TMA issue from one warp is slow)
constexpr int kTcThreads = (9 + kLoaderWarps) * 32;   // 2 softmax warpgroups, MMA issuer
constexpr int kTileBytes = kBlock * kHeadDim * 2;
constexpr int kTcSmemBytes = 7 * kTileBytes + 1024;

// Q tile layout ("half-interleaved", K-major, 128-byte swizzle): rows in
// groups of 8; a group holds its rows' columns 0..63 (1 KB, one swizzle atom)
// then columns 64..127 (1 KB), so one token's 8 rows x 128 columns are one
// contiguous 2 KB TMA box.  Byte offset of 16-byte chunk c of row r:
__device__ __forceinline__ uint32_t qmaj_off(int r, int c) {
  return (uint32_t)((r >> 3) * 2048 + (c >> 3) * 1024 + (r & 7) * 128 + (((c & 7) ^ (r & 7)) << 4));
}
// Descriptor of K step ks (16 columns) of that tile: 2 KB between 8-row groups.
__device__ __forceinline__ uint64_t qstep_desc(uint32_t base, int ks) {
  return sdesc_sw128_sbo(base + (uint32_t)((ks >> 2) * 1024 + (ks & 3) * 32), 2048);
}

struct PrefillArgs {
  int Hkv, Hq, G, S, B, NB;
  float scale_log2;                // softmax_scale * k_scale * log2(e)
  float v_scale;                   // applied to the normalised partial rows
  const __nv_bfloat16* q;
  const int32_t* row_ptr;
  const int32_t* q_idx;
  const uint8_t* k_pool;           // NVFP4: the pools, read with bulk copies (no tensor map)
  const uint8_t* v_pool;
};

// NVFP4 slots: per (page, KV head) a key slot (2h) and a value slot (2h + 1)
// of 128 rows x 72 bytes (64 bytes of E2M1 codes, 8 E4M3 block scales).
constexpr int kFp4Slot = kBlock * kFp4Row;

// NVFP4 slot in shared memory -> the 128 x 128 tile as TMA would have landed
// it (two 64-column halves, 128-byte swizzle): keys as bf16 (the S MMA's
// operand type, the queries being bf16), values as fp16 (the P V MMA's).
// e2m1 x e4m3 is exact in both (at most 6 significant bits, 2^-10 .. 2688).
// Values of rows past the last visible key become 0 (their scale byte may
// be anything, NaN included).  256 threads, four 16-element blocks each.
template <bool kValues>
__device__ __forceinline__ void fp4_slot_to_tile(const uint8_t* slot, uint8_t* tile, int ntok,
                                                 int tid) {
#pragma unroll
  for (int i = tid; i < kBlock * 8; i += 256) {
    const int key = i >> 3, c16 = i & 7;       // 16-element block c16 of row key
    const uint8_t* rp = slot + key * kFp4Row;
    const uint2 w = *reinterpret_cast<const uint2*>(rp + 8 * c16);
    const uint32_t sc = e4m3_scale_f16x2(rp[kHeadDim / 2 + c16]);
    uint32_t h[8];
    {
      uint32_t lo[4], hi[4];
      e2m1x8_to_f16x2(w.x, lo);
      e2m1x8_to_f16x2(w.y, hi);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        h[e] = hmul2_u32(lo[e], sc);
        h[4 + e] = hmul2_u32(hi[e], sc);
      }
    }
    if (kValues) {
      if (key >= ntok) {
#pragma unroll
        for (int e = 0; e < 8; ++e) h[e] = 0u;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const __nv_bfloat162 b =
            __float22bfloat162_rn(__half22float2(*reinterpret_cast<const __half2*>(&h[e])));
        h[e] = *reinterpret_cast<const uint32_t*>(&b);
      }
    }
    // elements 16 c16 .. + 7 and + 8 .. + 15: 16-byte chunks 2 c16, 2 c16 + 1
    *reinterpret_cast<uint4*>(tile + swz_tma(key, 2 * c16)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(tile + swz_tma(key, 2 * c16 + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

// Persistent: one CTA per SM walks the work items.  Per CSR row (KV head h,
// request r, key block j) the K tile and the V tile arrive by TMA (the next
// row's V during the current item, into the second V buffer; its K once the
// current item's last S has read the K tile); V is converted to fp16 in
// place and read by O = P V as an MN-major B operand.  M-tiles alternate
// between the two softmax warpgroups; warpgroup w's k-th tile (counted over
// the whole kernel) goes through
//   loaders: Q_k rows -> Q[w] (TMA)  once S_{k-1} has read Q[w]      (q_full)
//   issuer:  S_k = Q_k K^T (bf16) into TMEM region w, once Q_k landed and
//            O_{k-1} = P_{k-1} V has finished reading P_{k-1}      (s_ready)
//   WG:      S_k -> registers (thread = row), causal mask, softmax; P_k
//            (fp16) written over S_k's first 64 TMEM columns      (p_ready)
//   issuer:  O_k = P_k V (A operand from TMEM, fp16)                (o_ready)
//   WG:      O_k -> normalised fp16 row -> staging tile w (swizzled) ->
//            TMA tile stores into the partials, LSE beside them.
// TMEM: per warpgroup 128 columns of S / P and 128 of O (512 in all).  P
// never touches shared memory.  The issuer polls both warpgroups and serves
// whichever is ready, each O = P V before any S (P V completion gates the
// warpgroup's epilogue and its next S); the loaders run ahead across items.
template <bool FP4>
__global__ void __launch_bounds__(kTcThreads, 1)
prefill_tc_kernel(WsView ws, PrefillArgs a, const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v,
                  const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_o,
                  const __grid_constant__ CUtensorMap tmap_o8, int64_t rows) {
  extern __shared__ __align__(16) uint8_t tc_smem_raw[];
  // swizzled operand tiles want 1 KB alignment: round the base up (the
  // launch asks for 1 KB of slack)
  uint8_t* smem = tc_smem_raw + ((1024u - (smem_u32(tc_smem_raw) & 1023u)) & 1023u);
  uint8_t* Kt = smem;                          // K tile, bf16, K-major SW128 [key][d]
  // V of the current row and of the next one, [key][d] as TMA lands it; the
  // current one converted to fp16 in place is the MN-major B operand of P V
  // (NVFP4: one V buffer; the next row's two slots land in 18 KB of the second)
  auto Vb = [&](int i) { return i && !FP4 ? smem + 6 * kTileBytes : smem + kTileBytes; };
  uint8_t* Stg = smem + 6 * kTileBytes;        // NVFP4: key slot, value slot
  uint8_t* Pb = smem + 2 * kTileBytes;         // O staging tiles [2], fp16 [row][d]
  uint8_t* Qb = Pb + 2 * kTileBytes;           // Q[2], bf16 [row][d]

  __shared__ __align__(8) uint64_t k_full, v_full, k_free, vt_ready, q_full[2], s_ready[2],
      p_ready[2], o_ready[2];
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool issuer = warp == 8, loader = warp >= 9;
  const int lw = warp - 9;                     // loader warp index
  const int wg = warp >> 2;                    // softmax warpgroup (0, 1)
  const int wtid = tid & 127;                  // = this thread's row / TMEM lane
  if (tid == 0) {
    mbar_init(&k_full, 1);
    mbar_init(&v_full, 1);
    mbar_init(&k_free, 1);
    mbar_init(&vt_ready, 256);                 // the softmax warps, after the V conversion
    for (int w = 0; w < 2; ++w) {
      mbar_init(&q_full[w], kLoaderWarps);
      mbar_init(&s_ready[w], 1);
      mbar_init(&p_ready[w], 128);
      mbar_init(&o_ready[w], 1);
    }
    fence_barrier_init();
  }
  if (issuer) {
    tmem_alloc(&tmem_base, 512);               // S and O for each warpgroup
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  griddep_launch_dependents();
  griddep_wait();

  const int G = a.G, TPT = kBlock / G;         // tokens per M-tile
  const int lgG = __ffs(G) - 1;                // G divides 16
  const int n_items = ws.sched[rows];
  const uint32_t idesc_s = idesc_f16(1, 128, 128), idesc_o = idesc_f16_bmn(0, 128, 128);
  uint32_t k_phase = 0, v_phase = 0, kf_phase = 0, vt_phase = 0;
  int pf_row = -1;                             // issuer: row whose K / V are on the way
  int vsel = 1;                                // buffer of the current row's V (flips per row)
  int kS[2] = {0, 0}, kP[2] = {0, 0};          // issuer: S / PV issued per warpgroup
  int kL0 = 0, kL1 = 0;                        // loader: Q tiles loaded per warpgroup
  int kW = 0;                                  // warpgroup: tiles done
  int cur_row = -1;
  int n_kload = 0, n_vload = 0;                // issuer: K / V loads issued (drain on exit)
  // K / V tiles of CSR row rw: K into the K tile, V into V buffer `buf`
  auto load_k = [&](int rw) {
    ++n_kload;
    const int jj = rw % a.NB, rr = (rw / a.NB) % a.B, hh = rw / (a.NB * a.B);
    const int pg = ws.block_table[(int64_t)rr * a.NB + jj];
    const int y = ((pg < 0 ? 0 : pg) * a.Hkv + hh) * kBlock;
    mbar_arrive_expect_tx(&k_full, kTileBytes);
    const uint64_t pol = l2_evict_first_policy();   // one item's use, then gone
    tma_load_2d_hint(Kt, &tmap_k, 0, y, &k_full, pol);
    tma_load_2d_hint(Kt + kTileBytes / 2, &tmap_k, 64, y, &k_full, pol);
  };
  // NVFP4: both slots of CSR row rw into the staging area (on v_full)
  auto load_kv4 = [&](int rw) {
    ++n_vload;
    const int jj = rw % a.NB, rr = (rw / a.NB) % a.B, hh = rw / (a.NB * a.B);
    const int pg = ws.block_table[(int64_t)rr * a.NB + jj];
    const int64_t slot = ((int64_t)(pg < 0 ? 0 : pg) * a.Hkv + hh) * 2;
    mbar_arrive_expect_tx(&v_full, 2 * kFp4Slot);
    bulk_load(Stg, a.k_pool + slot * kFp4Slot, kFp4Slot, &v_full);
    bulk_load(Stg + kFp4Slot, a.v_pool + (slot + 1) * kFp4Slot, kFp4Slot, &v_full);
  };
  auto load_v = [&](int rw, int buf) {
    if (FP4) {
      load_kv4(rw);
      return;
    }
    ++n_vload;
    uint8_t* Vst = Vb(buf);
    const int jj = rw % a.NB, rr = (rw / a.NB) % a.B, hh = rw / (a.NB * a.B);
    const int pg = ws.block_table[(int64_t)rr * a.NB + jj];
    const int y = ((pg < 0 ? 0 : pg) * a.Hkv + hh) * kBlock;
    mbar_arrive_expect_tx(&v_full, kTileBytes);
    const uint64_t pol = l2_evict_first_policy();
    tma_load_2d_hint(Vst, &tmap_v, 0, y, &v_full, pol);
    tma_load_2d_hint(Vst + kTileBytes / 2, &tmap_v, 64, y, &v_full, pol);
  };
  // row of the next item of this CTA if it will be processed and needs other
  // K / V than `rw`, else -1 (issuer only)
  auto next_row = [&](int kk, int rw) {
    if (kk + (int)gridDim.x >= n_items) return -1;
    const int4 nit = ws.item_order[kk + gridDim.x];
    const int nr = nit.x;
    if (nr == rw) return -1;
    const int nj = nr % a.NB, nrr = (nr / a.NB) % a.B;
    if (ws.block_table[(int64_t)nrr * a.NB + nj] < 0 || nit.y >= nit.z) return -1;
    return nr;
  };
  for (int k = blockIdx.x; k < n_items; k += gridDim.x) {
    const int4 item = ws.item_order[k];          // largest items first
    const int row = item.x, beg = item.y, end = item.z;
    const int j = row % a.NB, r = (row / a.NB) % a.B, h = row / (a.NB * a.B);
    const int page = ws.block_table[(int64_t)r * a.NB + j];
    if (page < 0 || beg >= end) continue;      // flagged by the plan (uniform)
    const int ntok = min(kBlock, ws.req_seq_len[r] - j * kBlock);
    const int ntiles = (end - beg + TPT - 1) / TPT;

    // The loaders run ahead across items (their Q buffers are tracked per
    // tile); the others meet here once the previous item's MMAs are done.
    if (!loader) named_bar_sync(1, kTcThreads - 32 * kLoaderWarps);
    const bool new_row = row != cur_row;
    // A new row's K and V were prefetched during the previous item (K once its
    // last S had read the K tile); otherwise (first item, or the previous
    // item did not know) they are requested now.
    if (new_row) vsel ^= 1;
    if (new_row && issuer && lane == 0 && pf_row != row) {
      if (!FP4) load_k(row);
      load_v(row, vsel);
    }
    if (new_row && warp < 8 && FP4) {
      // NVFP4: the row's key and value slots -> the K tile (bf16) and the V
      // tile (fp16); the staging area is then free for the next row's slots
      mbar_wait(&v_full, v_phase, ws.hdr);
      v_phase ^= 1u;
      fp4_slot_to_tile<false>(Stg, Kt, ntok, tid);
      fp4_slot_to_tile<true>(Stg + kFp4Slot, Vb(0), ntok, tid);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&vt_ready);
    }
    if (new_row && warp < 8 && !FP4) {
      mbar_wait(&v_full, v_phase, ws.hdr);
      v_phase ^= 1u;
      {
        // V bf16 -> fp16 in place (16-byte chunks; a chunk lies in one key
        // row, 128 bytes per row and 64-column half); keys past the last
        // visible token become 0, whatever the page holds there
        uint8_t* vb = Vb(vsel);
        bool ovf = false;          // a value beyond the fp16 range
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int off = (tid + 256 * i) * 16;
          const int key = (off & (kTileBytes / 2 - 1)) >> 7;
          uint4 x = *reinterpret_cast<const uint4*>(vb + off);
          if (key >= ntok) {
            x = make_uint4(0u, 0u, 0u, 0u);
          } else {
            x.x = bf16x2_to_f16x2(x.x);
            x.y = bf16x2_to_f16x2(x.y);
            x.z = bf16x2_to_f16x2(x.z);
            x.w = bf16x2_to_f16x2(x.w);
            ovf |= f16x2_has_inf(x.x) | f16x2_has_inf(x.y) | f16x2_has_inf(x.z) |
                   f16x2_has_inf(x.w);
          }
          *reinterpret_cast<uint4*>(vb + off) = x;
        }
        if (__any_sync(0xffffffffu, ovf) && lane == 0) set_error(ws.hdr, MSA_DEVERR_FP16_RANGE);
        fence_proxy_async_smem();
      }
      // V (fp16) is ready for the PV MMAs; the issuer has meanwhile started
      // the item's S MMAs
      tc_fence_before();
      mbar_arrive(&vt_ready);
    }
    cur_row = row;

    if (loader) {
      // ------------------------------------------------------------ Q rows
      // Tile row rr is token rr / G, query head h * G + rr % G.  G >= 8: one
      // TMA box of G rows x 64 columns per token and half (1 KB-aligned in
      // the swizzled tile), completing on q_full[w] by transaction count;
      // rows of tokens past the end keep stale (finite) data, which the
      // softmax masks.  G < 8: 16-byte cp.async copies, 2 rows per instruction.
      // The loader warps share each tile's copies (box / instruction k goes to
      // warp k % kLoaderWarps) and each arrives on q_full[w] once.
      // each token's queries are read once per selected block (~20 times):
      // kept in L2 ahead of the K / V tiles and the streamed partials
      const uint64_t pol_q = l2_evict_last_policy();
      for (int t = 0; t < ntiles; ++t) {
        const int w = t & 1;
        const int n = w ? kL1 : kL0;
        if (n > 0) mbar_wait(&s_ready[w], (uint32_t)((n - 1) & 1), ws.hdr);
        const int e0 = beg + t * TPT;
        if (w) ++kL1; else ++kL0;
        if (G >= 8) {
          const int nt = min(TPT, end - e0);
          if (lane == 0) {
            if (lw == 0) mbar_arrive_expect_tx(&q_full[w], (uint32_t)(nt * G * 256));
            else mbar_arrive(&q_full[w]);
          }
          // box b: 8 rows (token b / (G / 8), rows 8 (b % (G / 8)) ...) x both
          // 64-column halves, one 2 KB group of the half-interleaved Q tile
          const int gpt = G >> 3;
          const int b = lane * kLoaderWarps + lw;
          if (b < nt * gpt) {
            const int tk = b / gpt, sub = b - tk * gpt;
            const int y = a.q_idx[e0 + tk] * a.Hq + h * G + 8 * sub;
            tma_load_3d_hint(Qb + w * kTileBytes + b * 2048, &tmap_q, 0, y, 0, &q_full[w], pol_q);
          }
          continue;
        }
        const uint32_t qdst = smem_u32(Qb + w * kTileBytes);
        int my_tok = -1;                         // G == 4: lane i < TPT holds token i
        if (lane < TPT && e0 + lane < end) my_tok = a.q_idx[e0 + lane];
#pragma unroll 2
        for (int i = lw; i < 64; i += kLoaderWarps) {
          const int rr = 2 * i + (lane >> 4);    // tile row: token rr / G, head rr % G
          const int c = lane & 15;
          int tk;
          if (TPT <= 32) {
            tk = __shfl_sync(0xffffffffu, my_tok, rr >> lgG);
          } else {
            const int e = e0 + (rr >> lgG);
            tk = e < end ? a.q_idx[e] : -1;
          }
          const __nv_bfloat16* src = a.q + ((int64_t)(tk < 0 ? 0 : tk) * a.Hq + h * G +
                                            (rr & (G - 1))) * kHeadDim + c * 8;
          cp_async16(qdst + qmaj_off(rr, c), src, tk < 0 ? 0 : 16);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_full[w]);
      }
      continue;
    }

    if (issuer) {
      if (lane == 0) {
        // descriptors of K step 0 (K tile, both Q buffers, this row's V);
        // step ks only moves the start address in the low word
        const uint64_t dk = kstep_desc(smem_u32(Kt), 0, 128);
        const uint64_t dq0 = qstep_desc(smem_u32(Qb), 0);
        const uint64_t dq1 = qstep_desc(smem_u32(Qb + kTileBytes), 0);
        const uint64_t dv = sdesc_sw128_mn(smem_u32(Vb(vsel)), kTileBytes / 2);
        const uint32_t vlo = (uint32_t)dv, vhi = (uint32_t)(dv >> 32);
        const uint32_t klo = (uint32_t)dk, khi = (uint32_t)(dk >> 32);
        const int nrow = next_row(k, row);
        if (new_row && !FP4) {
          mbar_wait(&k_full, k_phase, ws.hdr);
          k_phase ^= 1u;
        }
        bool vt_ok = !new_row;                   // V of this row converted
        // The next row's V goes to the other V buffer (the previous row's,
        // whose PV MMAs are done).  v_full counts one V load per phase, so it
        // is requested only once the softmax warps have seen this row's V land
        // (vt_ready): never two V loads in flight, never a phase they missed.
        bool v_done = nrow < 0;
        if (!v_done && vt_ok) {
          load_v(nrow, vsel ^ 1);
          v_done = true;
        }
        pf_row = nrow;
        bool k_done = nrow < 0 || FP4;           // the next row's K is requested
                                                 // (NVFP4: with its V, into the staging)
        int nS[2] = {0, 0}, nP[2] = {0, 0};      // this item's S / PV per warpgroup
        const int want[2] = {(ntiles + 1) / 2, ntiles / 2};
        uint32_t spins = 0;
        while (nP[0] < want[0] || nP[1] < want[1]) {
          bool did = false;
          // once this item's S MMAs have all completed, the next row's K
          if (!k_done && nS[0] == want[0] && nS[1] == want[1] &&
              mbar_test_wait(&k_free, kf_phase)) {
            load_k(nrow);
            k_done = true;
          }
          if (!vt_ok && mbar_test_wait(&vt_ready, vt_phase)) {
            vt_ok = true;
            vt_phase ^= 1u;
            tc_fence_after();
            if (!v_done) {
              load_v(nrow, vsel ^ 1);
              v_done = true;
            }
          }
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            if (vt_ok && nP[w] < nS[w] && mbar_test_wait(&p_ready[w], (uint32_t)(kP[w] & 1))) {
              tc_fence_after();
              // K step ks: P columns +8 ks, V rows 16 ks (+2 KB)
              const uint32_t ta = tbase + 256 * w, dt = ta + 128;
              umma_ts<false>(dt, ta, vlo, vhi, idesc_o);
#pragma unroll
              for (int ks = 1; ks < 8; ++ks)
                umma_ts<true>(dt, ta + 8 * ks, vlo + 128 * ks, vhi, idesc_o);
              umma_commit(&o_ready[w]);
              ++kP[w];
              ++nP[w];
              did = true;
            }
          }
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            // S_k overwrites P_{k-1}: only once O_{k-1} = P_{k-1} V completed
            if (nS[w] < want[w] && (!FP4 || vt_ok) &&
                mbar_test_wait(&q_full[w], (uint32_t)(kS[w] & 1)) &&
                (kS[w] == 0 || mbar_test_wait(&o_ready[w], (uint32_t)((kS[w] - 1) & 1)))) {
              tc_fence_after();
              const uint64_t dq = w ? dq1 : dq0;
              const uint32_t qlo = (uint32_t)dq, qhi = (uint32_t)(dq >> 32);
              const uint32_t dt = tbase + 256 * w;
              // K step ks: Q at +(ks / 4) KB + (ks % 4) 32 B, K at +(ks / 4) 16 KB + (ks % 4) 32 B
              umma_ss<false>(dt, qlo, qhi, klo, khi, idesc_s);
              umma_ss<true>(dt, qlo + 2, qhi, klo + 2, khi, idesc_s);
              umma_ss<true>(dt, qlo + 4, qhi, klo + 4, khi, idesc_s);
              umma_ss<true>(dt, qlo + 6, qhi, klo + 6, khi, idesc_s);
              umma_ss<true>(dt, qlo + 64, qhi, klo + 1024, khi, idesc_s);
              umma_ss<true>(dt, qlo + 66, qhi, klo + 1026, khi, idesc_s);
              umma_ss<true>(dt, qlo + 68, qhi, klo + 1028, khi, idesc_s);
              umma_ss<true>(dt, qlo + 70, qhi, klo + 1030, khi, idesc_s);
              umma_commit(&s_ready[w]);
              ++kS[w];
              ++nS[w];
              if (nS[0] == want[0] && nS[1] == want[1]) umma_commit(&k_free);   // last S
              did = true;
            }
          }
          if (did) {
            spins = 0;
          } else if (++spins > 16u * kWaitLimit) {  // bounded like every other wait
            atomicOr(&ws.hdr->err, MSA_DEVERR_TIMEOUT);
            break;
          }
        }
        // k_free completes once per item: consume it (and request K if the
        // loop ended first)
        mbar_wait(&k_free, kf_phase, ws.hdr);
        kf_phase ^= 1u;
        if (!k_done) load_k(nrow);
        if (!vt_ok) {                            // only on a timeout above
          mbar_wait(&vt_ready, vt_phase, ws.hdr);
          vt_phase ^= 1u;
        }
        if (!v_done) load_v(nrow, vsel ^ 1);
      }
      __syncwarp();
      continue;
    }

    // ---------------------------------------------------- softmax warpgroups
    uint8_t* prow = Pb + wg * kTileBytes;
    // the partials are read back only by the combine: evict them from L2
    // first, so they do not push out the queries that later items reuse
    const uint64_t pol_out = l2_evict_first_policy();
    const uint32_t tlane = tbase + ((uint32_t)(32 * (warp & 3)) << 16) + 256 * wg;
    const bool leader = wtid == 0;                  // issues the warpgroup's output stores
    // this thread's row of tile t: its token (< 0 past the end of the item)
    auto token_of = [&](int t) {
      const int e = beg + t * TPT + (wtid >> lgG);
      return t < ntiles && e < end ? a.q_idx[e] : -1;
    };
    int tok = token_of(wg), ntk = token_of(wg + 2);
    int pos = tok >= 0 ? ws.tok_pos[tok] : -1;
    for (int t = wg; t < ntiles; t += 2) {
      const int ftk = token_of(t + 4);              // two tiles ahead
      const int npos = ntk >= 0 ? ws.tok_pos[ntk] : -1;
      const bool valid = tok >= 0;
      const int lim = valid ? min(ntok, pos - j * kBlock + 1) : 0;

      mbar_wait(&s_ready[wg], (uint32_t)(kW & 1), ws.hdr);
      tc_fence_after();
      // pass 1: row max (raw scores).  The causal mask / the end of the
      // sequence only cut the diagonal / last block: a warp whose rows all see
      // the whole block skips the per-element mask.
      const bool full = __all_sync(0xffffffffu, lim >= kBlock);
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
      for (int cb = 0; cb < 2; ++cb) {
        uint32_t rg[64];
        tmem_ld64(tlane + 64 * cb, rg);
        tmem_ld_wait();
        if (full) {
#pragma unroll
          for (int i = 0; i < 64; i += 8) {
            mx[0] = fmax3(mx[0], __uint_as_float(rg[i]), __uint_as_float(rg[i + 1]));
            mx[1] = fmax3(mx[1], __uint_as_float(rg[i + 2]), __uint_as_float(rg[i + 3]));
            mx[2] = fmax3(mx[2], __uint_as_float(rg[i + 4]), __uint_as_float(rg[i + 5]));
            mx[3] = fmax3(mx[3], __uint_as_float(rg[i + 6]), __uint_as_float(rg[i + 7]));
          }
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            mx[i & 3] = fmaxf(mx[i & 3], 64 * cb + i < lim ? __uint_as_float(rg[i]) : -INFINITY);
        }
      }
      const float m = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      const float msc = m == -INFINITY ? 0.f : m * a.scale_log2;
      // pass 2: probabilities (exp2 domain, scale folded into one packed FMA),
      // fp16 P into TMEM over the S columns already read.  The exponent x <= 0
      // is rounded to fp16 and 2^x taken for two columns per special-function
      // instruction (fp16 is P's own precision); the row sum adds those same
      // fp16 values in fp32 (two pairs at a time in fp16, each term <= 1).
      // Masked columns (only outside the fast path) become -inf first.
      const uint64_t sc2 = f2(a.scale_log2, a.scale_log2), nm2 = f2(-msc, -msc);
      uint64_t ls2[4] = {0, 0, 0, 0};               // (+0.f, +0.f) pairs
#pragma unroll 1
      for (int cb = 0; cb < 2; ++cb) {
        uint32_t rg[64];
        tmem_ld64(tlane + 64 * cb, rg);
        tmem_ld_wait();
        if (!full) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (64 * cb + i >= lim) rg[i] = __float_as_uint(-INFINITY);
        }
        uint32_t pk[32];
#pragma unroll
        for (int i2 = 0; i2 < 32; i2 += 2) {
          float x0, x1, x2, x3;
          f2_split(fma_f2(f2u(rg[2 * i2], rg[2 * i2 + 1]), sc2, nm2), x0, x1);
          f2_split(fma_f2(f2u(rg[2 * i2 + 2], rg[2 * i2 + 3]), sc2, nm2), x2, x3);
          pk[i2] = ex2_f16x2(pack_f16(x0, x1));
          pk[i2 + 1] = ex2_f16x2(pack_f16(x2, x3));
          __half2 hs = __hadd2(*reinterpret_cast<const __half2*>(&pk[i2]),
                               *reinterpret_cast<const __half2*>(&pk[i2 + 1]));
          const float2 fs = __half22float2(hs);
          ls2[(i2 >> 1) & 3] = add_f2(ls2[(i2 >> 1) & 3], f2(fs.x, fs.y));
        }
        tmem_st32(tlane + 32 * cb, pk);             // keys 64cb.. -> columns 32cb..
      }
      float l;
      {
        float a0, a1;
        f2_split(add_f2(add_f2(ls2[0], ls2[1]), add_f2(ls2[2], ls2[3])), a0, a1);
        l = a0 + a1;
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_ready[wg]);

      // the staging tile still holds the previous tile's output until its
      // stores have read it
      if (leader) bulk_wait_read();
      named_bar_sync(2 + wg, 128);
      mbar_wait(&o_ready[wg], (uint32_t)(kW & 1), ws.hdr);
      tc_fence_after();
      // O_k -> normalised fp16 row, staged in the swizzled K-major layout.  The tile's rows are the
      // partial rows e0 * G ... of consecutive CSR entries, so the leader
      // stores them as TMA boxes: 128 rows for a full tile, 8-row boxes for
      // the last one, whose rows past a multiple of 8 (G < 8 only) their own
      // threads write.  tcgen05.ld is warp-collective: every lane loads.
      const float inv = l > 0.f ? a.v_scale / l : 0.f;
      const uint64_t inv2 = f2(inv, inv);
      const int e0 = beg + t * TPT;
      const int nrows = min(TPT, end - e0) * G;     // valid rows of this tile
      const bool tail_row = wtid >= (nrows & ~7) && wtid < nrows;
      __half* grow = static_cast<__half*>(ws.o_part) + ((int64_t)e0 * G + wtid) * kHeadDim;
#pragma unroll 1
      for (int cb = 0; cb < 2; ++cb) {
        uint32_t rg[64];
        tmem_ld64(tlane + 128 + 64 * cb, rg);
        tmem_ld_wait();
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
          uint32_t o4[4];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            float o0, o1;
            f2_split(mul_f2(f2u(rg[q8 * 8 + 2 * e2], rg[q8 * 8 + 2 * e2 + 1]), inv2), o0, o1);
            o4[e2] = pack_f16(o0, o1);
          }
          const uint4 v4 = make_uint4(o4[0], o4[1], o4[2], o4[3]);
          *reinterpret_cast<uint4*>(prow + kmaj_off(wtid, cb * 8 + q8, 128)) = v4;
          if (tail_row) reinterpret_cast<uint4*>(grow)[cb * 8 + q8] = v4;
        }
      }
      tc_fence_before();
      if (wtid < nrows)
        ws.lse_part[(int64_t)e0 * G + wtid] = l > 0.f ? (msc + log2f(l)) * kLn2 : -INFINITY;
      fence_proxy_async_smem();
      named_bar_sync(2 + wg, 128);
      if (leader) {
        if (nrows == kBlock) {
          tma_store_2d_hint(&tmap_o, 0, e0 * G, prow, pol_out);
          tma_store_2d_hint(&tmap_o, 64, e0 * G, prow + kTileBytes / 2, pol_out);
        } else {
          for (int b8 = 0; b8 < (nrows >> 3); ++b8) {
            tma_store_2d(&tmap_o8, 0, e0 * G + 8 * b8, prow + 1024 * b8);
            tma_store_2d(&tmap_o8, 64, e0 * G + 8 * b8, prow + kTileBytes / 2 + 1024 * b8);
          }
        }
        bulk_commit();
      }
      ++kW;
      tok = ntk;
      pos = npos;
      ntk = ftk;
    }
  }
  if (warp < 8) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  // Every MMA and copy has been waited for on the normal path.  After a wait
  // timed out some may still run: the issuer waits for its MMAs, and the
  // threads that issued TMA loads wait for the last phase they armed on each
  // barrier of those loads (bounded, no early exit), before the TMEM is freed
  // and the shared memory released.
  if (issuer && lane == 0) {
    umma_commit(&k_free);
    mbar_drain(&k_free, kf_phase);
  }
  if (*reinterpret_cast<volatile int*>(&ws.hdr->err) & MSA_DEVERR_TIMEOUT) {
    if (issuer && lane == 0) {
      if (n_kload > 0) mbar_drain(&k_full, (uint32_t)((n_kload - 1) & 1));
      if (n_vload > 0) mbar_drain(&v_full, (uint32_t)((n_vload - 1) & 1));
    }
    if (loader && lw == 0 && lane == 0 && G >= 8) {   // the Q boxes (G < 8 copies completed)
      if (kL0 > 0) mbar_drain(&q_full[0], (uint32_t)((kL0 - 1) & 1));
      if (kL1 > 0) mbar_drain(&q_full[1], (uint32_t)((kL1 - 1) & 1));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (issuer) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// First work item of every CSR row: ceil(row size / tokens per item), scanned.
__global__ void __launch_bounds__(256)
sched_count_kernel(const int32_t* __restrict__ row_ptr, int32_t* __restrict__ sched, int64_t rows,
                   int tok_per_item) {
  griddep_launch_dependents();
  griddep_wait();
  for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < rows; i += (int64_t)gridDim.x * 256) {
    const int n = row_ptr[i + 1] - row_ptr[i];
    sched[i + 1] = (n + tok_per_item - 1) / tok_per_item;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) sched[0] = 0;
}

// The work items request by request (requests ascending), largest first
// within a request (a counting sort in one CTA per request in turn).  A
// request's queries (tokens x H_q rows of 256 bytes, contiguous) are what the
// tiles re-read once per selected block: taken a request at a time they stay
// in L2, where all requests' together would not.  Largest first keeps the
// CTAs' round-robin shares of each request even.
__global__ void __launch_bounds__(1024)
item_order_kernel(const int32_t* __restrict__ row_ptr, WsView ws, int64_t rows, int tok_per_item,
                  int tpt, int B, int NB) {
  __shared__ int cnt[kTilesPerItem + 1], base[kTilesPerItem + 1];
  __shared__ int run_s;
  griddep_launch_dependents();
  griddep_wait();
  const int tid = threadIdx.x;
  auto items_of = [&](int64_t row, auto&& fn) {
    const int n = row_ptr[row + 1] - row_ptr[row];
    for (int k = 0; k * tok_per_item < n; ++k) {
      const int m = min(tok_per_item, n - k * tok_per_item);
      fn(k, (m + tpt - 1) / tpt);
    }
  };
  // rows (h, r, j) = (h * B + r) * NB + j; request r owns H_kv * NB of them
  const int64_t per_req = rows / B;
  auto row_of = [&](int r, int64_t i) { return ((i / NB) * B + r) * (int64_t)NB + i % NB; };
  if (tid == 0) run_s = 0;
  for (int r = 0; r < B; ++r) {
    if (tid <= kTilesPerItem) cnt[tid] = 0;
    __syncthreads();
    for (int64_t i = tid; i < per_req; i += 1024)
      items_of(row_of(r, i), [&](int, int sz) { atomicAdd(&cnt[sz], 1); });
    __syncthreads();
    if (tid == 0) {
      int run = run_s;
      for (int sz = kTilesPerItem; sz >= 0; --sz) {
        base[sz] = run;
        run += cnt[sz];
      }
      run_s = run;
    }
    __syncthreads();
    for (int64_t i = tid; i < per_req; i += 1024) {
      const int64_t row = row_of(r, i);
      const int rb = row_ptr[row], re = row_ptr[row + 1];
      items_of(row, [&](int k, int sz) {
        const int b = rb + k * tok_per_item;
        ws.item_order[atomicAdd(&base[sz], 1)] = make_int4((int)row, b, min(re, b + tok_per_item), 0);
      });
    }
    __syncthreads();
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
  const int NB = cfg->max_blocks_per_req, B = cfg->max_batch, Hkv = cfg->num_kv_heads;
  const int64_t wpr = csr_words_per_row(*cfg);
  const int64_t entries = (int64_t)max_tokens_of(*cfg) * Hkv * S;
  const int egrid = (int)std::min<int64_t>((entries + 255) / 256, 8 * 1024);
  if (cudaMemsetAsync(v.csr_bits, 0, 4 * (size_t)csr_words_of(*cfg), s) != cudaSuccess)
    return MSA_ERR_CUDA;
  if ((st = launch_pdl(csr_mark_kernel, dim3(egrid), dim3(256), 0, s, v, Hkv, NB, S, wpr,
                       selected)) != MSA_OK)
    return st;
  if ((st = launch_pdl(csr_count_kernel, dim3(grid), dim3(256), 0, s, v, Hkv, B, NB, wpr,
                       row_ptr)) != MSA_OK)
    return st;
  if ((st = launch_pdl(csr_scan_kernel, dim3(1), dim3(1024), 0, s, row_ptr, rows)) != MSA_OK)
    return st;
  if ((st = launch_pdl(csr_fill_kernel, dim3(egrid), dim3(256), 0, s, v, Hkv, B, NB, S, wpr,
                       selected, (const int32_t*)row_ptr, q_indices)) != MSA_OK)
    return st;
  // work schedule of msa_sparse_prefill: items of up to 16 M-tiles per row
  const int G = cfg->num_q_heads / cfg->num_kv_heads;
  const int tok_per_item = kTilesPerItem * (kBlock / G);
  const unsigned sgrid = (unsigned)((rows + 255) / 256 < 1024 ? (rows + 255) / 256 : 1024);
  if ((st = launch_pdl(sched_count_kernel, dim3(sgrid), dim3(256), 0, s, (const int32_t*)row_ptr,
                       v.sched, rows, tok_per_item)) != MSA_OK)
    return st;
  if ((st = launch_pdl(csr_scan_kernel, dim3(1), dim3(1024), 0, s, v.sched, rows)) != MSA_OK)
    return st;
  return launch_pdl(item_order_kernel, dim3(1), dim3(1024), 0, s, (const int32_t*)row_ptr, v, rows,
                    tok_per_item, kBlock / G, B, NB);
}

extern "C" msa_status msa_sparse_prefill(const msa_config* cfg, void* ws, const void* q,
                                         const void* k_pages, const void* v_pages,
                                         const int32_t* selected, const int32_t* row_ptr,
                                         const int32_t* q_indices, msa_stream_t stream) {
  msa_status st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (!is_prefill(*cfg)) return MSA_ERR_INVALID_ARG;
  const bool fp4 = cfg->kv_dtype == MSA_KV_NVFP4;
  if (cfg->kv_dtype != MSA_KV_BF16 && !fp4) return MSA_ERR_UNSUPPORTED;   // e4m3: not in prefill
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
  a.scale_log2 = cfg->softmax_scale * (fp4 ? cfg->k_scale : 1.f) * kLog2e;
  a.v_scale = fp4 ? cfg->v_scale : 1.f;
  a.k_pool = (const uint8_t*)k_pages;
  a.v_pool = (const uint8_t*)v_pages;
  a.q = (const __nv_bfloat16*)q;
  a.row_ptr = row_ptr;
  a.q_idx = q_indices;
  (void)selected;   // the CSR build recorded each entry's slot in ws
  const int64_t prow = (int64_t)cfg->num_pages * a.Hkv * kBlock;
  if (prow > 0x7fffffff) return MSA_ERR_UNSUPPORTED;
  CUtensorMap tk, tv, tq;
  if (fp4) {
    memset(&tk, 0, sizeof(tk));      // bulk copies from the pool pointers instead
    memset(&tv, 0, sizeof(tv));
  } else if (!make_pool_map(&tk, k_pages, prow, false) ||
             !make_pool_map(&tv, v_pages, prow, false)) {
    return MSA_ERR_CUDA;
  }
  // queries as [half (2)][row (tokens * H_q)][64 columns]: a box of 8 rows x
  // both halves is one 2 KB group of the half-interleaved Q tile (G >= 8)
  {
    const int64_t dims[3] = {64, (int64_t)max_tokens_of(*cfg) * a.Hq, 2};
    const int64_t str[2] = {(int64_t)kHeadDim * 2, 128};
    const int box[3] = {64, 8, 2};
    if (!make_bf16_map(&tq, q, 3, dims, str, box)) return MSA_ERR_CUDA;
  }
  // fp16 partial rows [T * H_q * S, 128] (2-byte elements, copied as bits):
  // whole M-tiles and 8-row boxes
  const int64_t orows = (int64_t)max_tokens_of(*cfg) * a.Hq * a.S;
  if (orows > 0x7fffffff) return MSA_ERR_UNSUPPORTED;
  CUtensorMap to, to8;
  const void* o_part = view_of(*cfg, ws).o_part;
  if (!make_pool_map(&to, o_part, orows, false) || !make_pool_map(&to8, o_part, orows, false, 8))
    return MSA_ERR_CUDA;
  const size_t smem = kTcSmemBytes;
  const int grid = sm_count();
  if (grid <= 0) return MSA_ERR_CUDA;
  auto kern = fp4 ? prefill_tc_kernel<true> : prefill_tc_kernel<false>;
  if ((st = set_smem(kern, smem)) != MSA_OK) return st;
  return launch_pdl(kern, dim3(grid), dim3(kTcThreads), smem, (cudaStream_t)stream,
                    view_of(*cfg, ws), a, tk, tv, tq, to, to8, rows);
}
