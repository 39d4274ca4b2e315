// msa_sparse_decode_noalloc: the sparse-decode step (plan -> split-K decode ->
// combine) for callers that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is not an option -- inside a
// host framework whose allocator owns every byte of device memory and forbids
// foreign allocations, inside a serving loop that has reserved almost all of
// HBM for its KV cache up front, or on a latency-critical path where an
// allocation (and the device synchronisation cudaMalloc / cudaFree may imply)
// is not acceptable.  Such a caller still owns its inputs and outputs; only the
// step's scratch (plan metadata, the validated block table and the split-K
// partials) lives in a fixed device array inside this library.
//
// The array is a file-scope __device__ buffer of MSA_NOALLOC_SCRATCH_BYTES;
// every GPU that loads the library holds it until the process exits.  Host
// code cannot use the array's name as a device address, so the first call on
// each device looks the address up with cudaGetSymbolAddress (with that device
// current) and caches it; every later call on that device reuses it.
#include <mutex>

#include "msa_internal.cuh"

namespace msa {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MSA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch on the current device (set up once).
msa_status scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MSA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return MSA_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return MSA_OK;
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" msa_status msa_sparse_decode_noalloc(const msa_config* cfg, int32_t batch,
                                                const int32_t* seq_lens,
                                                const int32_t* block_table, int32_t bt_stride,
                                                const void* q, const void* k_pages,
                                                const void* v_pages, const int32_t* selected,
                                                void* out, float* lse, msa_stream_t stream) {
  msa_status st = check_config(cfg);
  if (st != MSA_OK) return st;
  if (layout_of(*cfg).total > (size_t)MSA_NOALLOC_SCRATCH_BYTES) return MSA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != MSA_OK) return st;
  // The plan clears the scratch header (the error word) and rewrites every
  // metadata field the decode reads; the decode writes every partial the
  // combine reads, so nothing left by an earlier call is ever used.
  if ((st = msa_plan(cfg, batch, seq_lens, nullptr, block_table, bt_stride, scratch, stream)) !=
      MSA_OK)
    return st;
  if ((st = msa_sparse_decode(cfg, scratch, q, k_pages, v_pages, selected, stream)) != MSA_OK)
    return st;
  return msa_combine(cfg, scratch, out, lse, stream);
}

extern "C" msa_status msa_noalloc_check_device_error(int32_t* flags, msa_stream_t stream) {
  if (flags == nullptr) return MSA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  msa_status st = scratch_address(&scratch);
  if (st != MSA_OK) return st;
  // The scratch starts with the same header and per-request plan words as a
  // workspace (zero before the first call: no error).
  return msa_check_device_error(scratch, flags, stream);
}
