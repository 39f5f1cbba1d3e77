// Failure-path check of the bounded device waits.
//
// One thread waits on an mbarrier that nothing ever arrives on, through the
// same bounded wait the grouped GEMM uses for its pipeline.  After limit_ns
// the wait gives up, records the timeout status in the device status word and
// the kernel returns normally, leaving the CUDA context usable.
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void bounded_wait_probe_kernel(int *status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, status, limit_ns);  // phase 0 never completes
}

}  // namespace

cudaError_t launch_bounded_wait_probe(int *status, uint64_t limit_ns, cudaStream_t stream) {
    bounded_wait_probe_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace moe
