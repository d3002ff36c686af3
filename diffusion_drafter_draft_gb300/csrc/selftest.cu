// Self-test of the bounded device-side waits: the same helpers the kernels use
// wait for something that is never signalled (an mbarrier nothing arrives on, a
// grid-barrier target one arrival above the CTAs that exist). Each must give up
// after the given limit, record DARTREE_ETIMEOUT in the status word and return,
// leaving the context usable. Nothing faults and nothing waits without bound.
#include "common.cuh"
#include "kernels.h"

namespace dartree {

__global__ void selftest_mbar_kernel(int* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival expected, none will come
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, status, limit_ns);
}

__global__ void selftest_grid_kernel(unsigned* ctr, int* status, uint64_t limit_ns) {
    __shared__ unsigned timed_out;
    if (threadIdx.x == 0) timed_out = 0;
    __syncthreads();
    // every CTA arrives once; the target counts one CTA more than the grid has
    grid_barrier(ctr, gridDim.x + 1u, status, &timed_out, limit_ns);
}

int launch_selftest_wait(int which, unsigned* ctr, int* status, uint64_t limit_ns, cudaStream_t stream) {
    if (which == 0) {
        selftest_mbar_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    } else {
        if (cudaMemsetAsync(ctr, 0, sizeof(unsigned), stream) != cudaSuccess) return DARTREE_ECUDA;
        selftest_grid_kernel<<<2, 32, 0, stream>>>(ctr, status, limit_ns);
    }
    return cudaGetLastError() == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

}  // namespace dartree
