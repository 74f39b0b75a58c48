// Self-test of the library's bounded mbarrier wait: a wait on a barrier that nothing
// arrives on must give up after its limit and leave the context usable; after one
// arrival the same wait must succeed at once.  Test infrastructure only.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_sm100.cuh"

using namespace kda::sm100;

// out[0]: 1 if the wait succeeded, 0 if it gave up; out[1]: ns spent in the wait (thread 0)
__global__ void __launch_bounds__(32, 1) wait_selftest_kernel(uint64_t limit_ns, int arrive,
                                                              unsigned long long* out)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncwarp();
    if (arrive && threadIdx.x == 0) mbar_arrive(&bar);
    __syncwarp();
    const uint64_t t0 = globaltimer_ns();
    const bool ok = mbar_wait_bounded(&bar, 0, limit_ns);
    const uint64_t t1 = globaltimer_ns();
    if (threadIdx.x == 0) {
        out[0] = ok ? 1ull : 0ull;
        out[1] = t1 - t0;
    }
}

extern "C" int wait_selftest(unsigned long long limit_ns, int arrive, void* out)
{
    wait_selftest_kernel<<<1, 32>>>(limit_ns, arrive, static_cast<unsigned long long*>(out));
    if (cudaGetLastError() != cudaSuccess) return -1;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : -2;
}
