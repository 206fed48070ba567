// Self-check of the bounded-wait error path. Every kernel of the library waits
// on mbarriers through mbar_wait, which gives up after about a second, records
// DSA_ERR_TIMEOUT in the caller's status word and lets the kernel return. This
// entry point runs that same wait on a barrier that either receives its one
// arrival or receives none, so a caller can see the error reach the host with
// the context still usable -- without any fault, trap or endless loop.
#include "common.cuh"

namespace dsa {

__global__ void __launch_bounds__(32) wait_selftest_kernel(int32_t arrive, int32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (arrive) mbar_arrive(&bar);
        mbar_wait(&bar, 0, &abort_flag, status);
    }
}

}  // namespace dsa

extern "C" int dsa_bounded_wait_selftest(int32_t arrive, int32_t *dev_status, void *stream) {
    if (!dev_status) return DSA_ERR_ARG;
    dsa::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(arrive, dev_status);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
