// Failure-detection self-test: one CTA runs the kernels' bounded mbarrier wait
// on a barrier that nothing ever arrives at, with a caller-chosen short limit.
// The wait gives up, records the timeout in the device status word and the
// kernel returns: no GPU fault, the context stays usable.
#include "fa_internal.h"
#include "fa_ptx.cuh"

#include "fa.h"

namespace fa {
namespace {

__global__ void __launch_bounds__(32) fa_selftest_wait_kernel(int* status, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);   // one arrival expected; none ever comes
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, status, timeout_ns);
}

// One thread runs a bounds check whose condition is false (no memory is
// touched): an FA_DEBUG build records FA_DEV_BOUNDS in the status word.
__global__ void __launch_bounds__(32) fa_selftest_bounds_kernel(int* status) {
  if (threadIdx.x == 0) {
    volatile uint32_t col = 512;   // one column past the allocation
    if (FA_DBG_OK(status, tmem_in(col, 32))) { /* the access a check guards would go here */ }
  }
}

}  // namespace
}  // namespace fa

extern "C" int fa_debug_build(void) {
#ifdef FA_DEBUG
  return 1;
#else
  return 0;
#endif
}

extern "C" int fa_selftest_bounds(void* stream) {
#ifndef FA_DEBUG
  (void)stream;
  return FA_ERR_UNSUPPORTED;
#else
  int* status = fa::device_status_ptr();
  if (!status) return fa::cuda_fail(cudaGetLastError());
  const cudaError_t e = fa::launch_kernel(fa::fa_selftest_bounds_kernel, dim3(1), dim3(32), 0,
                                          static_cast<cudaStream_t>(stream), status);
  return e == cudaSuccess ? FA_OK : fa::cuda_fail(e);
#endif
}

extern "C" int fa_selftest_wait_timeout(unsigned long long timeout_ns, void* stream) {
  if (timeout_ns == 0 || timeout_ns > 10000000000ull) return FA_ERR_INVALID_ARG;
  int* status = fa::device_status_ptr();
  if (!status) return fa::cuda_fail(cudaGetLastError());
  const cudaError_t e = fa::launch_kernel(fa::fa_selftest_wait_kernel, dim3(1), dim3(32), 0,
                                          static_cast<cudaStream_t>(stream), status, timeout_ns);
  return e == cudaSuccess ? FA_OK : fa::cuda_fail(e);
}
