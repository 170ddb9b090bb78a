// Failure-detection self-test: proves on the device that a bounded wait on a
// barrier that never completes gives up, records an error code the host can
// read, and leaves the context usable.  Nothing faults, traps or hangs.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace gemm {

namespace {

__global__ void selftest_wait_kernel(int* err, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);  // expects one arrival that no thread will make
        abort_flag = 0u;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) wait_bounded(b, 0u, &abort_flag, err, kDevErrTimeoutSelfTest, timeout_ns);
    __syncthreads();
}

}  // namespace

cudaError_t launch_selftest_wait(int* err, uint64_t timeout_ns, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(err, timeout_ns);
    return cudaGetLastError();
}

}  // namespace gemm
