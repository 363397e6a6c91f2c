// selftest.cu -- a kernel whose bounded wait is meant to run out.
//
// Every wait of this library's kernels on an mbarrier is bounded: after kWaitTimeoutNs it
// records PGQA_DEV_TIMEOUT (and where it gave up) in the device status word and returns,
// so a lost arrival ends in an error status the host reads instead of a hung GPU.  The
// kernel here waits, with that same function, on a barrier that nothing arrives at, so
// that the failure path can be checked end to end: the status word, the diagnostic
// record, the status call that clears them, and a context that stays usable.
#include "ptx.cuh"

namespace pgqa {
namespace selftest {

__global__ void __launch_bounds__(32) expired_wait_kernel(int* status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncwarp();
    // nothing arrives on `bar`, so its phase 0 never completes and the wait gives up
    if (threadIdx.x == 0) mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, status);
    __syncwarp();
}

cudaError_t launch_expired_wait(int* status, cudaStream_t stream) {
    expired_wait_kernel<<<1, 32, 0, stream>>>(status);
    return cudaGetLastError();
}

}  // namespace selftest
}  // namespace pgqa
