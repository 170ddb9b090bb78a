// Test-only producer kernel: lets the kernels behind it in the stream launch
// at once (griddepcontrol.launch_dependents), waits delay_ns of %globaltimer
// time (bounded by an iteration cap as well), then copies src to dst.  A
// consumer launched with programmatic stream serialization may therefore
// start while this kernel has not yet written dst; it must wait for this
// kernel (griddepcontrol.wait) before reading dst.
#include <cuda_runtime.h>

#include <cstdint>

__global__ void late_writer_kernel(uint4* dst, const uint4* src, int64_t n16, uint64_t delay_ns) {
    asm volatile("griddepcontrol.launch_dependents;" :::);
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (uint32_t it = 0; it < (1u << 24); ++it) {
        uint64_t t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > delay_ns) break;
    }
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        dst[i] = src[i];
}

extern "C" int late_writer(void* dst, const void* src, int64_t bytes, uint64_t delay_ns, void* stream) {
    if (bytes % 16 != 0 || (reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) % 16 != 0) return -1;
    // 8 CTAs: the kernels behind it find most SMs free and start there while
    // this kernel waits (a full-size grid would keep them off the SMs)
    late_writer_kernel<<<8, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4*>(dst), static_cast<const uint4*>(src), bytes / 16, delay_ns);
    return static_cast<int>(cudaGetLastError());
}
