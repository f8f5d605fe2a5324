// selftest.cu -- checks of the kernels' failure path that fault nothing: one thread waits,
// through the same bounded waits the kernels use, on something nothing completes (an
// mbarrier, as every GEMM role waits; a global counter, as the ring forward's producers
// wait). The wait gives up after the given wall time, records MOK_ERR_TIMEOUT in the device
// status word and the kernel returns, leaving the context usable.
#include "common.cuh"
#include "mok_internal.h"
#include "tc.cuh"

namespace mok {
namespace {

__global__ void bounded_wait_probe_kernel(int *status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        abort_flag = 0;
        tc::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // no thread arrives on the barrier, so its phase 0 never completes
        tc::wait_bounded(&bar, 0u, status, &abort_flag, limit_ns);
    }
}

// a counter that nothing raises
__device__ int32_t g_never_raised;

__global__ void bounded_count_probe_kernel(int *status, uint64_t limit_ns) {
    __shared__ int abort_flag;
    if (threadIdx.x == 0) abort_flag = 0;
    __syncthreads();
    if (threadIdx.x == 0)
        tc::wait_count_bounded(&g_never_raised, 1, status, &abort_flag, limit_ns);
}

}  // namespace

cudaError_t launch_bounded_count_probe(int *status, uint64_t limit_ns, cudaStream_t s) {
    bounded_count_probe_kernel<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_bounded_wait_probe(int *status, uint64_t limit_ns, cudaStream_t s) {
    bounded_wait_probe_kernel<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace mok
