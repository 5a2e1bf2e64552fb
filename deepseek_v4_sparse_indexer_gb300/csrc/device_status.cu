// Exercises the device-side failure path without a fault: one thread waits on
// an mbarrier that nothing ever completes, gives up after a bounded time and
// reports DS4A_DEV_TIMEOUT in the device status word, exactly as the bounded
// waits of the compute kernels do when a producer never arrives.
#include "common.cuh"
#include "internal.h"

namespace ds4a {
namespace {

__global__ void __launch_bounds__(32) debug_wait_kernel(uint32_t *status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&bar, 0)) {
            if (globaltimer_ns() - t0 > limit_ns) {
                report(status, DS4A_DEV_TIMEOUT);
                break;
            }
        }
    }
}

}  // namespace

cudaError_t launch_debug_wait(uint32_t *status, unsigned long long limit_ns, cudaStream_t s) {
    debug_wait_kernel<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace ds4a
