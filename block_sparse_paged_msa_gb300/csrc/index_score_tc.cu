// Index scores of a decode / speculative-verify step on the tensor cores:
// for each request r, KV head h, visible block j and each of r's q_len new
// tokens t,
//   score[t, h, j] = max over the keys k of block j at positions <= pos(t) of
//                    idx_q[t, h, :] . idx_k[k, h, :]
// (the definition of msa_index_score; vLLM sparse_attention_msa.py runs
// regular decode and speculative verification with decode_query_len new
// tokens per request, sglang minimax_sparse_backend.py hands idx_q and the
// index-K cache to the sparse decode op).
//
// Why a second kernel: with q_len tokens sharing each index-key tile the SIMT
// scan (index_score.cu) needs q_len x d / 8 registers per lane for the
// queries, which at q_len = 4 leaves two CTAs per SM and too few bytes in
// flight for the HBM stream.  Here the tile stream is decoupled from the
// registers:
//  * work item = (request, block, KV head): one 128-key tile of the HND
//    index-key pool (32 KiB at d = 128), contiguous, read once per step;
//  * a persistent CTA per SM; warp 0 resolves 32 items at a time (a lane
//    each) and, one lane issuing, streams each item's tile and the request's
//    query rows (16 rows: the q_len tokens and whatever follows them, zero
//    past the step) with TMA into a ring of ~180 KB of shared memory;
//  * warp 1 issues tcgen05.mma with the keys as M = 128 rows, the query rows
//    as N = 16 and K = d, bf16 in, fp32 accumulators in TMEM (two 16-column
//    buffers) -- the products are exact for the integer-valued index vectors;
//  * warps 2-5 read the accumulators (thread = key row), mask keys past each
//    token's position, and reduce the maxima across the block's 128 rows.
#include <mutex>

#include "tcgen05.cuh"

namespace msa {
namespace {

constexpr int kThreads = 192;     // producer, MMA issuer, 4 epilogue warps
constexpr int kQRows = 16;        // MMA N: a request's query tokens, padded

template <int DIDX>
struct TcCfg {
  static constexpr int kTile = kBlock * DIDX * 2;     // index-key tile (MMA A)
  static constexpr int kQTile = kQRows * DIDX * 2;    // query rows (MMA B)
  static constexpr int kStage = kTile + kQTile;       // a multiple of 1 KiB
  static constexpr int kStages = DIDX == 128 ? 5 : 10;
  static constexpr int kHalves = DIDX / 64;           // 64-column TMA boxes
  static constexpr int kSmem = kStages * kStage + 1024;
  static_assert(kStage % 1024 == 0, "stages must keep the 1 KiB swizzle atoms aligned");
};

// An item as the producer publishes it with its stage.
struct TcItem {
  int qs, j, h, page;
  int lim[4];          // keys of the block visible to token qs + i (0: not this request's)
};

struct TcArgs {
  int Hkv, max_blocks, max_tokens;
  float* scores;
};

template <int DIDX, int QL>
__global__ void __launch_bounds__(kThreads, 1)
index_score_tc_kernel(WsView ws, TcArgs a, const __grid_constant__ CUtensorMap tmap_q,
                      const __grid_constant__ CUtensorMap tmap_k) {
  using C = TcCfg<DIDX>;
  extern __shared__ __align__(16) uint8_t tc_smem_raw[];
  uint8_t* smem = tc_smem_raw + ((1024u - (smem_u32(tc_smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t full[C::kStages], empty[C::kStages], acc_full[2],
      acc_empty[2];
  __shared__ TcItem meta[C::kStages];
  __shared__ float red[2][4][4];
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1 + 4);     // the MMA's commit + the 4 epilogue warps
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  griddep_launch_dependents();
  griddep_wait();

  const int batch = ws.hdr->batch;
  const int total = ws.hdr->total_blocks * a.Hkv;
  const int n_my = total > (int)blockIdx.x ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    uint32_t loaded = 0;         // lane 0: stages whose latest item issued copies
    for (int base = 0; base < n_my; base += 32) {
      // lane l resolves this CTA's item base + l
      TcItem mine;
      {
        const int k = base + lane;
        const int item = (int)blockIdx.x + k * (int)gridDim.x;
        mine.page = -1;
        mine.qs = mine.j = mine.h = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) mine.lim[i] = 0;
        if (k < n_my) {
          const int h = item % a.Hkv, b = item / a.Hkv;
          int lo = 0, hi = batch - 1;   // request of flat block b
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (ws.req_cu_nb[mid] <= b) lo = mid; else hi = mid - 1;
          }
          const int j = b - ws.req_cu_nb[lo];
          const int qs = ws.req_qstart[lo];
          mine.qs = qs;
          mine.j = j;
          mine.h = h;
          mine.page = ws.block_table[(int64_t)lo * a.max_blocks + j];
#pragma unroll
          for (int i = 0; i < QL; ++i) {
            // a request owns QL consecutive tokens; anything else is left unscored
            const bool own = qs + i < a.max_tokens && ws.tok_req[qs + i] == lo;
            const int lim = own ? ws.tok_pos[qs + i] - j * kBlock + 1 : 0;
            mine.lim[i] = lim > kBlock ? kBlock : (lim < 0 ? 0 : lim);
          }
        }
      }
      const int nb = min(32, n_my - base);
      for (int l = 0; l < nb; ++l) {
        TcItem it;
        it.qs = __shfl_sync(0xffffffffu, mine.qs, l);
        it.j = __shfl_sync(0xffffffffu, mine.j, l);
        it.h = __shfl_sync(0xffffffffu, mine.h, l);
        it.page = __shfl_sync(0xffffffffu, mine.page, l);
#pragma unroll
        for (int i = 0; i < 4; ++i) it.lim[i] = __shfl_sync(0xffffffffu, mine.lim[i], l);
        if (lane == 0) {
          const int k = base + l, s = k % C::kStages;
          mbar_wait(&empty[s], (uint32_t)(((k / C::kStages) & 1) ^ 1), ws.hdr);
          meta[s] = it;
          if (it.page >= 0) {
            uint8_t* st = smem + s * C::kStage;
            mbar_arrive_expect_tx(&full[s], (uint32_t)C::kStage);
            const int y = (it.page * a.Hkv + it.h) * kBlock;
#pragma unroll
            for (int x = 0; x < C::kHalves; ++x) {
              tma_load_2d(st + x * (C::kTile / C::kHalves), &tmap_k, 64 * x, y, &full[s]);
              tma_load_3d(st + C::kTile + x * (C::kQTile / C::kHalves), &tmap_q, 64 * x, it.h,
                          it.qs, &full[s]);
            }
            loaded |= 1u << s;
          } else {
            // a page the plan flagged: nothing to load, the epilogue writes -inf
            mbar_arrive(&full[s]);
            loaded &= ~(1u << s);
          }
        }
        __syncwarp();
      }
    }
    if (lane == 0 && (*reinterpret_cast<volatile int*>(&ws.hdr->err) & MSA_DEVERR_TIMEOUT)) {
      // a wait gave up somewhere: let this CTA's copies land before it retires
      // (the last phase of a stage completes once every copy armed on it has)
      for (int s = 0; s < C::kStages; ++s)
        if ((loaded >> s) & 1u) {
          const int last = (n_my - 1 - s) / C::kStages;   // phase of the stage's last item
          mbar_drain(&full[s], (uint32_t)(last & 1));
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(1, 128, kQRows);
      for (int k = 0; k < n_my; ++k) {
        const int s = k % C::kStages, b = k & 1;
        mbar_wait(&full[s], (uint32_t)((k / C::kStages) & 1), ws.hdr);
        mbar_wait(&acc_empty[b], (uint32_t)(((k >> 1) & 1) ^ 1), ws.hdr);
        tc_fence_after();
        if (meta[s].page >= 0) {
          const uint32_t as = smem_u32(smem + s * C::kStage);
          const uint32_t bs = as + C::kTile;
#pragma unroll
          for (int ks = 0; ks < DIDX / 16; ++ks)
            umma_f16(tbase + 16 * b, kstep_desc(as, ks, kBlock), kstep_desc(bs, ks, kQRows), idesc,
                     ks > 0);
          umma_commit(&empty[s]);
          umma_commit(&acc_full[b]);
        } else {
          mbar_arrive(&empty[s]);
          mbar_arrive(&acc_full[b]);
        }
      }
      // the last accumulators are waited for by the epilogue; after a timeout
      // wait for this thread's MMAs before TMEM is released
      if (n_my > 0 && (*reinterpret_cast<volatile int*>(&ws.hdr->err) & MSA_DEVERR_TIMEOUT)) {
        const int k = n_my - 1;
        mbar_drain(&acc_full[k & 1], (uint32_t)((k >> 1) & 1));
      }
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;                         // TMEM lanes 32q .. 32q + 31
    const int row = 32 * q + lane;                  // key row of the block
    const uint32_t tl = tbase + ((uint32_t)(32 * q) << 16);
    for (int k = 0; k < n_my; ++k) {
      const int s = k % C::kStages, b = k & 1;
      mbar_wait(&full[s], (uint32_t)((k / C::kStages) & 1), ws.hdr);   // meta[s] is published
      const TcItem it = meta[s];
      mbar_wait(&acc_full[b], (uint32_t)((k >> 1) & 1), ws.hdr);
      tc_fence_after();
      uint32_t acc[4];
      tmem_ld4(tl + 16 * b, acc);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&acc_empty[b]);
        mbar_arrive(&empty[s]);
      }
#pragma unroll
      for (int i = 0; i < QL; ++i) {
        float x = it.page >= 0 && row < it.lim[i] ? __uint_as_float(acc[i]) : -INFINITY;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
        if (lane == 0) red[b][q][i] = x;
      }
      named_bar_sync(1, 128);
      if (q == 0 && lane < QL && it.lim[lane] > 0) {
        const float m = fmaxf(fmaxf(red[b][0][lane], red[b][1][lane]),
                              fmaxf(red[b][2][lane], red[b][3][lane]));
        a.scores[((int64_t)(it.qs + lane) * a.Hkv + it.h) * a.max_blocks + it.j] = m;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 32);
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

template <int DIDX, int QL>
msa_status launch_tc(const msa_config& c, const WsView& v, const void* idx_q, const void* idx_k,
                     float* scores, cudaStream_t s) {
  using Cf = TcCfg<DIDX>;
  const int T = max_tokens_of(c);
  TcArgs a;
  a.Hkv = c.num_kv_heads;
  a.max_blocks = c.max_blocks_per_req;
  a.max_tokens = T;
  a.scores = scores;
  // idx_q as [T][H_kv][d]: boxes of 64 columns x 1 head x 16 tokens (zero past T)
  CUtensorMap tq, tk;
  {
    const int64_t dims[3] = {DIDX, c.num_kv_heads, T};
    const int64_t str[2] = {(int64_t)DIDX * 2, (int64_t)c.num_kv_heads * DIDX * 2};
    const int box[3] = {64, 1, kQRows};
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
  msa_status st = set_smem(index_score_tc_kernel<DIDX, QL>, Cf::kSmem);
  if (st != MSA_OK) return st;
  const int grid = sm_count();
  if (grid <= 0) return MSA_ERR_CUDA;
  return launch_pdl(index_score_tc_kernel<DIDX, QL>, dim3(grid), dim3(kThreads),
                    (size_t)Cf::kSmem, s, v, a, tq, tk);
}

}  // namespace

msa_status decode_index_score_tc(const msa_config& c, const WsView& v, const void* idx_q,
                                 const void* idx_k, float* scores, cudaStream_t s) {
  const bool d128 = c.index_dim == 128;
  switch (c.q_len) {
    case 1: return d128 ? launch_tc<128, 1>(c, v, idx_q, idx_k, scores, s)
                        : launch_tc<64, 1>(c, v, idx_q, idx_k, scores, s);
    case 2: return d128 ? launch_tc<128, 2>(c, v, idx_q, idx_k, scores, s)
                        : launch_tc<64, 2>(c, v, idx_q, idx_k, scores, s);
    case 3: return d128 ? launch_tc<128, 3>(c, v, idx_q, idx_k, scores, s)
                        : launch_tc<64, 3>(c, v, idx_q, idx_k, scores, s);
    case 4: return d128 ? launch_tc<128, 4>(c, v, idx_q, idx_k, scores, s)
                        : launch_tc<64, 4>(c, v, idx_q, idx_k, scores, s);
    default: return MSA_ERR_UNSUPPORTED;
  }
}

}  // namespace msa
