// selftest.cu -- exercises the bounded-wait path of the kernels on the GPU
// without a fault: one thread waits on an mbarrier phase that nothing ever
// completes, gives up after the kernels' wait limit (2 s of %globaltimer),
// sets the device error word as a timed-out GEMV wait does, and returns.
#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {

namespace {

__global__ void selftest_wait_timeout_kernel(unsigned *err) {
    __shared__ __align__(8) unsigned long long bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_barrier_init();
    // nobody arrives: phase 0 never completes, the bounded wait gives up
    if (!mbar_wait_bounded(b, 0)) atomicOr(err, kDevErrTimeoutFull);
}

}  // namespace

cudaError_t launch_selftest_wait_timeout(unsigned *err, cudaStream_t stream) {
    selftest_wait_timeout_kernel<<<1, 32, 0, stream>>>(err);
    return cudaGetLastError();
}

}  // namespace nvfp4
