// Failure-detection check: a wait on an mbarrier that nothing arrives at,
// bounded in SM clock cycles exactly like the waits of the tensor-core
// kernels, which then reports through the device error word and returns.
#include "kda_internal.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace {

__global__ void __launch_bounds__(32, 1) wait_timeout_kernel(long long limit_cycles, int32_t* dev_err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);   // one arrival expected; none ever comes
    tc::fence_mbar_init();
  }
  __syncwarp();
  const bool ok = tc::mbar_wait(&bar, 0, limit_cycles);
  if (__any_sync(0xffffffffu, !ok) && threadIdx.x == 0) atomicExch(dev_err, (int32_t)kDevErrTimeout);
}

}  // namespace
}  // namespace kda

extern "C" KDA_API kda_status kda_check_wait_timeout(int64_t limit_cycles, cudaStream_t stream) {
  if (limit_cycles < 1 || limit_cycles > 1000000000LL) return KDA_ERR_INVALID_ARG;
  int32_t* dev_err = nullptr;
  if (kda::device_error_ptr(&dev_err) != cudaSuccess) return KDA_ERR_CUDA;
  kda::wait_timeout_kernel<<<1, 32, 0, stream>>>((long long)limit_cycles, dev_err);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
