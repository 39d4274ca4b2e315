// Prefill index scores on fifth-generation tensor cores: for every query token
// t of a prefill chunk, KV head h and key block j visible to t,
//   score[t, h, j] = max over the keys k of block j at positions <= pos(t) of
//                    idx_q[t, h, :] . idx_k[k, h, :]
// (the same definition as the decode scan, with the causal limit of each
// token).  vLLM minimax_m3/nvidia/sparse_attention_msa.py
// (MiniMaxM3SparseMSAImpl.forward) takes the per-token block selection of a
// prefill chunk as input; sglang minimax_sparse_backend.py
// (MiniMaxSparseAttnBackend.forward_extend) hands idx_q and the index-K cache
// to the prefill op.  The score formula is this library's specification: max
// over tokens, fp32 accumulation (exact for integer-valued index vectors).
//
// A chunk's scores are a dense causal GEMM, [tokens x d] x [d x keys], reduced
// by a max over each 128-key block: tensor-core work.  Design:
//  * work unit = (KV head h, 128-token tile m of the step's tokens, chunk c of
//    the key blocks); the tile may hold the tail of one request and the head
//    of the next (segments), each against its own blocks;
//  * a persistent CTA per SM: warp 0 issues TMA (the tile's idx_q rows once per
//    unit through a 3-D map [T][H_kv][d]; pairs of index-key pages into a ring
//    of stages), warp 1 issues tcgen05.mma M = 128 tokens x N = 256 keys (two
//    blocks) x K = d, bf16 in, fp32 accumulators in TMEM (two 256-column
//    buffers), warps 2-5 read the accumulators (thread = token) and write the
//    per-block causal maxima;
//  * units are ordered tile-fastest, so the CTAs running at one time read the
//    same index-key pages and share them through L2.
#include <algorithm>
#include <mutex>

#include "tcgen05.cuh"

namespace msa {
namespace {

constexpr int kIdxThreads = 192;        // producer, MMA issuer, 4 epilogue warps
constexpr int kIdxTile = 128;           // tokens per unit (MMA M)

template <int DIDX>
struct IdxCfg {
  static constexpr int kATile = kIdxTile * DIDX * 2;          // idx_q tile bytes
  static constexpr int kPage = kBlock * DIDX * 2;             // one index-key page tile
  static constexpr int kStage = 2 * kPage;                    // a pair of pages (N = 256)
  static constexpr int kStages = DIDX == 128 ? 3 : 6;
  static constexpr int kHalves = DIDX / 64;                   // 64-column TMA boxes
  static constexpr int kSmem = kATile + kStages * kStage + 1024;
};

struct IdxArgs {
  int Hkv, NB, MT, NC, kc;   // KV heads, blocks per request, token tiles, chunks, blocks/chunk
  float* scores;
};

// Segments of token tile [t0, t1): runs of tokens of one request.  For each
// segment with work in chunk c, fn(r, s, e, jb, je) gets the request, the
// segment's tokens [s, e) and its blocks [jb, je).  Tokens of no request
// (idle / flagged) are skipped.
template <typename F>
__device__ __forceinline__ void for_segments(const WsView& ws, int t0, int t1, int c, int kc,
                                             F&& fn) {
  int s = t0;
  while (s < t1) {
    const int r = ws.tok_req[s];
    if (r < 0) {
      ++s;
      continue;
    }
    const int e = min(t1, ws.req_qstart[r + 1]);
    const int nb = min(ws.tok_pos[e - 1] / kBlock + 1, ws.req_nb[r]);
    const int jb = c * kc, je = min(jb + kc, nb);
    if (jb < je) fn(r, s, e, jb, je);
    s = e;
  }
}

template <int DIDX>
__global__ void __launch_bounds__(kIdxThreads, 1)
prefill_index_tc_kernel(WsView ws, IdxArgs a, const __grid_constant__ CUtensorMap tmap_q,
                        const __grid_constant__ CUtensorMap tmap_k) {
  using C = IdxCfg<DIDX>;
  extern __shared__ __align__(16) uint8_t idx_smem_raw[];
  uint8_t* smem = idx_smem_raw + ((1024u - (smem_u32(idx_smem_raw) & 1023u)) & 1023u);
  uint8_t* At = smem;
  uint8_t* Bst = smem + C::kATile;
  __shared__ __align__(8) uint64_t full[C::kStages], empty[C::kStages], acc_full[2],
      acc_empty[2], a_full, a_empty;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 128);
    }
    mbar_init(&a_full, 1);
    mbar_init(&a_empty, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  griddep_launch_dependents();
  griddep_wait();

  const int T = ws.hdr->num_tokens;
  const int n_units = a.Hkv * a.NC * a.MT;
  int pairs = 0, units = 0;   // pairs of blocks / units with work, this CTA so far
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const int m = u % a.MT, c = (u / a.MT) % a.NC, h = u / (a.MT * a.NC);
    const int t0 = m * kIdxTile;
    if (t0 >= T) continue;
    const int t1 = min(T, t0 + kIdxTile);
    int npairs = 0;
    for_segments(ws, t0, t1, c, a.kc,
                 [&](int, int, int, int jb, int je) { npairs += (je - jb + 1) >> 1; });
    if (npairs == 0) continue;   // uniform: every role skips the unit

    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        if (units > 0) mbar_wait(&a_empty, (uint32_t)((units - 1) & 1), ws.hdr);
        mbar_arrive_expect_tx(&a_full, C::kATile);
#pragma unroll
        for (int x = 0; x < C::kHalves; ++x)
          tma_load_3d(At + x * (C::kATile / C::kHalves), &tmap_q, 64 * x, h, t0, &a_full);
        int it = pairs;
        for_segments(ws, t0, t1, c, a.kc, [&](int r, int, int, int jb, int je) {
          for (int j = jb; j < je; j += 2, ++it) {
            const int s = it % C::kStages;
            mbar_wait(&empty[s], (uint32_t)(((it / C::kStages) & 1) ^ 1), ws.hdr);
            const int np = min(2, je - j);
            mbar_arrive_expect_tx(&full[s], (uint32_t)(np * C::kPage));
            uint8_t* st = Bst + s * C::kStage;
            for (int p = 0; p < np; ++p) {
              const int page = ws.block_table[(int64_t)r * a.NB + j + p];
              const int y = ((page < 0 ? 0 : page) * a.Hkv + h) * kBlock;
#pragma unroll
              for (int x = 0; x < C::kHalves; ++x)
                tma_load_2d(st + x * (C::kStage / C::kHalves) + p * (C::kPage / C::kHalves),
                            &tmap_k, 64 * x, y, &full[s]);
            }
          }
        });
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_f16(1, 128, 256);
        mbar_wait(&a_full, (uint32_t)(units & 1), ws.hdr);
        tc_fence_after();
        const uint32_t as = smem_u32(At);
        int it = pairs;
        for_segments(ws, t0, t1, c, a.kc, [&](int, int, int, int jb, int je) {
          for (int j = jb; j < je; j += 2, ++it) {
            const int s = it % C::kStages, b = it & 1;
            mbar_wait(&full[s], (uint32_t)((it / C::kStages) & 1), ws.hdr);
            mbar_wait(&acc_empty[b], (uint32_t)(((it >> 1) & 1) ^ 1), ws.hdr);
            tc_fence_after();
            const uint32_t bs = smem_u32(Bst + s * C::kStage);
#pragma unroll
            for (int ks = 0; ks < DIDX / 16; ++ks)
              umma_f16(tbase + 256 * b, kstep_desc(as, ks, 128), kstep_desc(bs, ks, 256), idesc,
                       ks > 0);
            umma_commit(&empty[s]);
            umma_commit(&acc_full[b]);
          }
        });
        umma_commit(&a_empty);   // the tile's last MMA has read A
      }
      __syncwarp();
    } else {
      // ------------------------------------------------------------ epilogue
      const int row = 32 * (warp & 3) + lane;    // TMEM lane = token of the tile
      const int t = t0 + row;
      const int my_r = t < t1 ? ws.tok_req[t] : -1;
      const int pos = my_r >= 0 ? ws.tok_pos[t] : -1;
      float* srow = a.scores + ((int64_t)t * a.Hkv + h) * a.NB;
      const uint32_t tl = tbase + ((uint32_t)(32 * (warp & 3)) << 16);
      int it = pairs;
      for_segments(ws, t0, t1, c, a.kc, [&](int r, int, int, int jb, int je) {
        const bool mine = my_r == r;
        for (int j = jb; j < je; j += 2, ++it) {
          const int b = it & 1;
          mbar_wait(&acc_full[b], (uint32_t)((it >> 1) & 1), ws.hdr);
          tc_fence_after();
          float best[2];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            // keys of block j + q visible to this row (<= 0: none, >= 128: all)
            const int lim = mine ? pos - (j + q) * kBlock + 1 : 0;
            const bool whole = __all_sync(0xffffffffu, lim >= kBlock);
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
            for (int cb = 0; cb < 2; ++cb) {
              uint32_t rg[64];
              tmem_ld64(tl + 256 * b + 128 * q + 64 * cb, rg);
              tmem_ld_wait();
              if (whole) {
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
                  mx[i & 3] =
                      fmaxf(mx[i & 3], 64 * cb + i < lim ? __uint_as_float(rg[i]) : -INFINITY);
              }
            }
            best[q] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
          }
          tc_fence_before();
          mbar_arrive(&acc_empty[b]);
          if (mine && pos >= j * kBlock) srow[j] = best[0];
          if (mine && j + 1 < je && pos >= (j + 1) * kBlock) srow[j + 1] = best[1];
        }
      });
    }
    pairs += npairs;
    ++units;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <typename K>
msa_status set_idx_smem(K kernel, size_t bytes) {
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) ==
                 cudaSuccess
             ? MSA_OK
             : MSA_ERR_CUDA;
}

template <int DIDX>
msa_status launch_index(const msa_config& c, const WsView& v, const void* idx_q,
                        const void* idx_k, float* scores, cudaStream_t s) {
  using Cf = IdxCfg<DIDX>;
  const int T = max_tokens_of(c);
  IdxArgs a;
  a.Hkv = c.num_kv_heads;
  a.NB = c.max_blocks_per_req;
  a.MT = (T + kIdxTile - 1) / kIdxTile;
  a.NC = (a.NB + 63) / 64;
  a.kc = (a.NB + a.NC - 1) / a.NC;
  a.kc += a.kc & 1;                                   // whole pairs of blocks per chunk
  a.scores = scores;
  if ((int64_t)a.Hkv * a.NC * a.MT > 0x7fffffff) return MSA_ERR_UNSUPPORTED;
  // idx_q as [T][H_kv][d]: boxes of 64 columns x 1 head x 128 tokens
  CUtensorMap tq, tk;
  {
    const int64_t dims[3] = {DIDX, c.num_kv_heads, T};
    const int64_t str[2] = {(int64_t)DIDX * 2, (int64_t)c.num_kv_heads * DIDX * 2};
    const int box[3] = {64, 1, kIdxTile};
    if (!make_bf16_map(&tq, idx_q, 3, dims, str, box)) return MSA_ERR_CUDA;
  }
  // index-key pool as [pages * H_kv * 128 rows][d]: boxes of 64 columns x 128 rows
  {
    const int64_t rows = (int64_t)c.num_pages * c.num_kv_heads * kBlock;
    if (rows > 0x7fffffff) return MSA_ERR_UNSUPPORTED;
    const int64_t dims[2] = {DIDX, rows};
    const int64_t str[1] = {(int64_t)DIDX * 2};
    const int box[2] = {64, kBlock};
    if (!make_bf16_map(&tk, idx_k, 2, dims, str, box)) return MSA_ERR_CUDA;
  }
  msa_status st = set_idx_smem(prefill_index_tc_kernel<DIDX>, Cf::kSmem);
  if (st != MSA_OK) return st;
  const int grid = sm_count();
  if (grid <= 0) return MSA_ERR_CUDA;
  return launch_pdl(prefill_index_tc_kernel<DIDX>, dim3(grid), dim3(kIdxThreads),
                    (size_t)Cf::kSmem, s, v, a, tq, tk);
}

}  // namespace

msa_status prefill_index_score(const msa_config& c, const WsView& v, const void* idx_q,
                               const void* idx_k, float* scores, cudaStream_t s) {
  if (!aligned16(idx_q) || !aligned16(idx_k)) return MSA_ERR_INVALID_ARG;
  return c.index_dim == 128 ? launch_index<128>(c, v, idx_q, idx_k, scores, s)
                            : launch_index<64>(c, v, idx_q, idx_k, scores, s);
}

}  // namespace msa
