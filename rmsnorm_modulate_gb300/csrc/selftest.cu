// Self-test of the bounded waits every TMA-fed kernel relies on: one warp
// waits on an mbarrier that nothing ever completes, with a caller-chosen
// limit, then records the timeout in this unit's device error word exactly
// as a real kernel would, and returns.  Nothing faults and nothing hangs; the
// host reads the error word (rmsmod_device_status) and the context stays
// usable.
#include "device_common.cuh"
#include "launch.h"
#include "selftest.h"

namespace rmsmod {

namespace {

__device__ unsigned int g_error;

__global__ void __launch_bounds__(32) wait_timeout_kernel(const unsigned long long limit_ns)
{
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1u);  // one arrival completes phase 0; none ever comes
        mbar_init_fence();
    }
    __syncwarp();
    if (!mbar_wait(b, 0u, limit_ns) && threadIdx.x == 0)
        atomicOr(&g_error, kErrCopyTimeout);
}

}  // namespace

cudaError_t launch_selftest_wait(unsigned long long limit_ns, cudaStream_t stream)
{
    wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

cudaError_t selftest_error(unsigned* bits, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_error, sizeof(unsigned));
    if (e == cudaSuccess && clear && *bits) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_error, &zero, sizeof(unsigned));
    }
    return e;
}

}  // namespace rmsmod
