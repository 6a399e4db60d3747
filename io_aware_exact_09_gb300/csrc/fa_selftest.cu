// fa_selftest.cu -- exercises the device-side failure path of the attention
// kernels on purpose, without a fault: one warp waits, with the kernels' own
// bounded wait (mbar_wait), on a barrier phase that nothing completes.  After
// FA_WAIT_TIMEOUT_NS the wait gives up, records FA_ERR_DEVICE_TIMEOUT and the
// wait site in the workspace status words and raises the CTA's abort flag; a
// second wait then returns at once through that flag, and the kernel exits
// normally, leaving the context usable.
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

namespace {

constexpr unsigned kSelftestSite = 0x5e1f;

__global__ void __launch_bounds__(32) fa_selftest_wait_kernel(unsigned *status, unsigned *result) {
    __shared__ __align__(8) uint64_t bar_storage;
    __shared__ int abort_flag;
    const uint32_t bar = smem_u32(&bar_storage);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);          // one arrival would complete phase 0; none comes
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncwarp();
    const Guard g{status, status + 1, &abort_flag};
    // 1: the timeout path; 2: the abort-flag path (returns without waiting out the limit)
    const bool first = mbar_wait_warp(bar, 0, g, kSelftestSite);
    const uint64_t t0 = globaltimer_ns();
    const bool second = mbar_wait_warp(bar, 0, g, kSelftestSite + 1);
    const uint64_t dt = globaltimer_ns() - t0;
    if (threadIdx.x == 0) {
        result[0] = first ? 1u : 0u;
        result[1] = second ? 1u : 0u;
        result[2] = dt < FA_WAIT_TIMEOUT_NS / 4 ? 1u : 0u;   // the second wait did not run to the limit
    }
}

}  // namespace

cudaError_t launch_selftest_wait(unsigned *status, unsigned *result, cudaStream_t st) {
    fa_selftest_wait_kernel<<<1, 32, 0, st>>>(status, result);
    return cudaGetLastError();
}

}  // namespace fa
