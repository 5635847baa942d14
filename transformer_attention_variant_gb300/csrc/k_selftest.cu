// k_selftest.cu -- exercises the bounded-wait failure path on the device without any
// fault: one CTA initialises an mbarrier that nothing will ever arrive on and waits on
// it with a short limit.  The wait must give up, record its site in the status word and
// let the kernel return normally.
#include "iha_internal.h"
#include "ptx.cuh"

namespace iha {

__global__ void wait_selftest_kernel(int *status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, status, kSiteSelfTest, &abort_flag, limit_ns);
    __syncthreads();
}

cudaError_t launch_wait_selftest(int *status, unsigned long long limit_ns, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace iha
