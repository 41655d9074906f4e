// diag.cu -- diagnostic kernels that exercise the library's failure paths
// without faulting the GPU.
//
// diag_wait_timeout_kernel runs the bounded mbarrier wait every pipelined
// kernel of the library uses, on a barrier that no thread ever arrives at and
// with no copy, tensor-core operation or tensor-memory allocation in flight:
// the wait gives up after the caller's limit, records MNB_ERR_TIMEOUT in the
// device error word and the kernel returns normally, so the context stays
// usable.
#include "common.cuh"
#include "kernels.h"

namespace mnb {

namespace {

__global__ void __launch_bounds__(32) diag_wait_timeout_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncwarp();
    // phase 0 needs one arrival; none comes
    warp_wait_for(&bar, 0, limit_ns);
}

}  // namespace

cudaError_t diag_take_error(unsigned int* out) { return take_unit_error(out); }

cudaError_t launch_diag_wait_timeout(uint64_t limit_ns, cudaStream_t stream) {
    diag_wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

}  // namespace mnb
