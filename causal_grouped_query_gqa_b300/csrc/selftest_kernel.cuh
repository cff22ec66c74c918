// selftest_kernel.cuh -- checks the failure detection of the kernels on the
// device itself, without faulting anything: one CTA whose two waiting threads
// wait on mbarriers that nothing ever arrives on.  The first gives up after a
// short budget, raises the CTA abort flag and records GQA_ERR_DEVICE_TIMEOUT in
// the status word; the second waits with the kernels' normal 2 s budget and
// must leave through the abort flag instead, within about one suspension
// (1 ms) of the first.  Both record how long they waited.
#pragma once

#include "sm100_ptx.cuh"

namespace gqa {
namespace selftest {

enum : int { kTimeoutCode = -9 };

__device__ unsigned long long g_selftest_elapsed_ns[2];
__device__ int g_selftest_returned[2];

__global__ void __launch_bounds__(64, 1) selftest_wait_kernel(int *status, uint64_t budget_ns) {
  __shared__ uint64_t bar[2];
  __shared__ AbortState ab;
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    ab.flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    const uint64_t t0 = globaltimer_ns();
    const bool ok = warp == 0 ? mbar_wait(&bar[0], 0, &ab, status, kTimeoutCode, budget_ns)
                              : mbar_wait(&bar[1], 0, &ab, status, kTimeoutCode);
    g_selftest_elapsed_ns[warp] = globaltimer_ns() - t0;
    g_selftest_returned[warp] = ok ? 1 : 0;
  }
}

}  // namespace selftest
}  // namespace gqa
