// selftest.cu -- a check, on the device, of the bounded waits every pipeline
// in this library uses: mbar_wait_bounded (the decode kernels' TMA stages)
// and tc_wait (the tcgen05 kernels' roles, which also give up once another
// role has aborted). Two threads each wait on an mbarrier expecting one
// arrival. With `arrive` set, that arrival is made first and both waits must
// return at once; without it nothing ever arrives, so each wait runs out
// after its cycle limit, sets PA_DEV_TIMEOUT in the status word and returns
// false, and the kernel ends normally: a stalled pipeline reports an error
// instead of hanging the GPU.
#include "prefill_tc.cuh"

namespace pagedkv {

__global__ void __launch_bounds__(64) wait_selftest_kernel(int arrive, uint32_t* status) {
    __shared__ uint64_t bars[2];
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (arrive && (threadIdx.x == 0 || threadIdx.x == 32)) mbar_arrive(&bars[threadIdx.x >> 5]);
    __syncthreads();
    bool ok = true;
    if (threadIdx.x == 0) ok = mbar_wait_bounded(&bars[0], 0u, status);
    if (threadIdx.x == 32) ok = tc_wait(&bars[1], 0u, status, &abort_flag);
    // a wait that returned without an arrival would be a missed timeout
    if (!arrive && ok && (threadIdx.x == 0 || threadIdx.x == 32) && status)
        atomicOr(status, PA_DEV_BAD_LEN);
}

cudaError_t launch_wait_selftest(int arrive, uint32_t* status, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 64, 0, stream>>>(arrive, status);
    return cudaGetLastError();
}

}  // namespace pagedkv
