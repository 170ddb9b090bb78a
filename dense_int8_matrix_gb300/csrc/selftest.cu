// The device error word and the failure-detection self-test.
//
// Every bounded wait in the library's kernels that gives up records its code
// in one int per device (first code wins; kernels only write it).  The word is
// a file-scope static __device__ variable, so no entry point allocates it and
// the allocating and allocation-free entry points share it; gemm_device_error
// reads and clears it.  In host code the variable's name is a host-side
// stand-in, so device_error_word() looks its device address up with
// cudaGetSymbolAddress (callers cache it per device).
//
// The self-test proves on the device that a bounded wait on a barrier that
// never completes gives up, records an error code the host can read, and
// leaves the context usable.  Nothing faults, traps or hangs.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace gemm {

namespace {

static __device__ int g_device_err;

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

cudaError_t device_error_word(int** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_device_err);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    *out = static_cast<int*>(p);
    return cudaSuccess;
}

cudaError_t launch_selftest_wait(int* err, uint64_t timeout_ns, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(err, timeout_ns);
    return cudaGetLastError();
}

}  // namespace gemm
