// Self-test of the bounded device-side wait (w4a16_selftest_wait_timeout).
//
// Every pipeline wait in the library's kernels goes through sm100::mbar_wait,
// which gives up after a wall-clock limit, raises the CTA's abort flag and
// writes W4A16_ERR_TIMEOUT to the caller's status word instead of hanging.
// That path only runs when something upstream is broken, so this entry point
// exercises it on purpose: one warp waits, with a short limit, on an mbarrier
// that nothing ever completes (a flag that nothing sets), and the kernel then
// returns normally, leaving the context usable.
#include "sm100.cuh"
#include "w4a16.h"
#include "w4a16_internal.h"

namespace w4a16 {
namespace {

__global__ void __launch_bounds__(32) wait_never_completed_kernel(int* dev_status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    sm100::mbar_init(&bar, 1);  // expects one arrival, which never comes
    abort_flag = 0;
    sm100::fence_mbar_init();
  }
  __syncwarp();
  (void)sm100::mbar_wait(&bar, 0, &abort_flag, dev_status, limit_ns);
}

}  // namespace
}  // namespace w4a16

extern "C" w4a16_status w4a16_selftest_wait_timeout(int* dev_status, unsigned long long limit_ns,
                                                    cudaStream_t stream) {
  if (dev_status == nullptr || limit_ns == 0 || limit_ns > 10000000000ull) return W4A16_ERR_INVALID_ARG;
  w4a16::wait_never_completed_kernel<<<1, 32, 0, stream>>>(dev_status, limit_ns);
  return cudaGetLastError() == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}
