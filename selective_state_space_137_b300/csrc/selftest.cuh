// selftest.cuh -- a kernel whose bounded wait can never complete, so that the
// timeout path of the device-side waits (error word + early return) can be
// exercised without hanging or faulting the GPU.
#pragma once
#include "tma.cuh"

namespace ssm {

__global__ void __launch_bounds__(32) wait_timeout_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);          // one arrival expected; nothing arrives
        fence_barrier_init();
    }
    __syncwarp();
    mbar_wait_bounded(&bar, 0, limit_ns);   // gives up after limit_ns, latches the error
}

}  // namespace ssm
