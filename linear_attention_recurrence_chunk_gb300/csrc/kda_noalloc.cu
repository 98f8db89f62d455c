// Allocation-free chunked prefill: kda_chunk_fwd with its scratch space taken
// from a fixed array that the library itself holds in device memory.
//
// Some callers cannot call cudaMalloc: a serving engine that reserves almost
// all device memory for its caches at start-up (a later allocation would fail
// or fragment its pool), a plug-in whose host owns the device allocator, or
// code that must run within a memory budget fixed before the first request.
// They still pass their own inputs and outputs; only the scratch space moves
// into this file.
//
// The scratch array is a file-scope __device__ array, so every GPU that loads
// this library holds KDA_NOALLOC_SCRATCH_BYTES of it until the process exits.
// In host code its name is only a stand-in for the symbol, not a device
// address, so the address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and then cached.  The cache
// assumes the device's primary context for the life of the process: after a
// cudaDeviceReset the module is loaded again and the cached address would be
// stale, so a caller that resets a device must not use this entry point on it
// afterwards.
//
// Nothing in the array has to start at zero: every byte that a call reads was
// written earlier in that same call (chunk map, then per-chunk records), so
// the contents left by the previous call do not matter.  All calls share the
// one array, so two calls whose work overlaps on the GPU (different streams,
// or different host threads) race on it and must not overlap.
#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr size_t kScratchBytes = (size_t)KDA_NOALLOC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_kda_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on the
// first call for that device, then cached).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_kda_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

kda_status kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const void* g, const float* beta,
                                 const float* initial_state, const int32_t* cu_seqlens, int32_t num_seqs, int64_t B,
                                 int64_t T, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt, void* o,
                                 float* final_state, cudaStream_t stream) {
  const size_t need = kda_chunk_fwd_workspace_size(B, T, H, d_k, d_v, num_seqs, dt);
  if (need == SIZE_MAX)   // invalid or unsupported shape: kda_chunk_fwd's own status, in its own order
    return kda_chunk_fwd(q, k, v, g, beta, initial_state, cu_seqlens, num_seqs, B, T, H, d_k, d_v, dt, o,
                         final_state, nullptr, 0, stream);
  if (need > kScratchBytes) return KDA_ERR_INVALID_ARG;   // problem too large for the fixed scratch array
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return KDA_ERR_CUDA;
  return kda_chunk_fwd(q, k, v, g, beta, initial_state, cu_seqlens, num_seqs, B, T, H, d_k, d_v, dt, o, final_state,
                       scratch, kScratchBytes, stream);
}

}  // extern "C"
