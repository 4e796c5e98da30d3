// Self test of the bounded barrier wait used by every pipelined kernel: one
// warp waits on an mbarrier phase that nothing will complete; the wait must
// give up after the limit and record a timeout in the status word, leaving the
// context usable.
#include <cuda_runtime.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {
__global__ void wait_selftest_kernel(int* status, unsigned long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    __syncwarp();
    if (threadIdx.x == 0 && !mbar_wait_bounded(b, 0, timeout_ns)) atomicOr(status, kDevErrTimeout);
}
}  // namespace

cudaError_t launch_wait_selftest(int* status, unsigned long long timeout_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace pa
