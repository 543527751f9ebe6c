// qmm_dbg_wait_timeout: exercises the bounded mbarrier wait that every kernel
// of the library uses, on a barrier that nothing ever arrives on, so that the
// time-out path (error code in the device error word, abort flag, normal
// return) can be tested without faulting or hanging the GPU.
#include "../../include/qmm.h"
#include "ptx.cuh"
#include "qmm_internal.h"

namespace qmm {

__global__ void __launch_bounds__(32) wait_timeout_probe_kernel(uint32_t* err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_word;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_word = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_for(&bar, 0, &abort_word, err, DEV_TIMEOUT_PROBE, limit_ns);
    __syncwarp();
}

cudaError_t launch_wait_timeout_probe(uint32_t* err, uint64_t limit_ns, cudaStream_t s) {
    wait_timeout_probe_kernel<<<1, 32, 0, s>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace qmm
