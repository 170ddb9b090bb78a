// Skinny int8 GEMM on CUDA cores (m <= 128, in launches of at most 64 rows;
// used when the tensor-core skinny kernel does not apply): C = A x B where B (stored K-major as Bt,
// n x k) is far larger than A, so the kernel's job is to stream Bt from HBM
// once.  The patent CN114238853A (claim 4 S3) notes that such shapes are too
// small to fill the chip with output tiles; here they get their own kernel.
//
// Mapping: a CTA owns 32 output columns j (one per lane) and all m rows of
// C.  Its 8 warps split K into interleaved 16-byte vectors, so the 8 warps of
// a CTA read consecutive 16-byte pieces of the same 128-byte lines of Bt.
// Each lane keeps m int32 partial sums (one per row of A), formed with dp4a
// on its own Bt row and the A vector that all lanes of the warp share (one
// broadcast load).  The warps' partial sums are added in shared memory
// (int32, exact) and written to C with coalesced stores.  This is the
// warp-level partial-sum scheme of "CUDA编程实践" §2 (reduce), with the
// final cross-warp sum in shared memory instead of shuffles.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace gemm {

namespace {

constexpr int kSkWarps = 8;
constexpr int kSkCols = 32;
constexpr int kSkUnroll = 8;

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

template <int MT>
__global__ void __launch_bounds__(kSkWarps * 32) skinny_dp4a_kernel(const int8_t* __restrict__ A,
                                                                    const int8_t* __restrict__ Bt,
                                                                    int32_t* __restrict__ C, int m, int64_t n,
                                                                    int64_t k) {
    __shared__ int32_t red[MT][kSkCols];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int t = threadIdx.x; t < MT * kSkCols; t += blockDim.x) (&red[0][0])[t] = 0;
    __syncthreads();

    const int64_t j = static_cast<int64_t>(blockIdx.x) * kSkCols + lane;
    const bool col_ok = j < n;
    const int8_t* brow = Bt + (col_ok ? j : 0) * k;
    const int64_t nvec = k / 16;

    int32_t acc[MT];
#pragma unroll
    for (int i = 0; i < MT; ++i) acc[i] = 0;

    for (int64_t v0 = warp; v0 < nvec; v0 += kSkWarps * kSkUnroll) {
        uint4 b[kSkUnroll];
#pragma unroll
        for (int u = 0; u < kSkUnroll; ++u) {
            const int64_t v = v0 + static_cast<int64_t>(u) * kSkWarps;
            b[u] = (v < nvec && col_ok) ? ld_stream16(brow + v * 16) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kSkUnroll; ++u) {
            const int64_t v = v0 + static_cast<int64_t>(u) * kSkWarps;
            if (v < nvec) {
#pragma unroll
                for (int i = 0; i < MT; ++i) {
                    if (i < m) {
                        const uint4 a = __ldg(reinterpret_cast<const uint4*>(A + static_cast<int64_t>(i) * k + v * 16));
                        int s = acc[i];
                        s = __dp4a(static_cast<int>(a.x), static_cast<int>(b[u].x), s);
                        s = __dp4a(static_cast<int>(a.y), static_cast<int>(b[u].y), s);
                        s = __dp4a(static_cast<int>(a.z), static_cast<int>(b[u].z), s);
                        s = __dp4a(static_cast<int>(a.w), static_cast<int>(b[u].w), s);
                        acc[i] = s;
                    }
                }
            }
        }
    }

#pragma unroll
    for (int i = 0; i < MT; ++i)
        if (i < m) atomicAdd(&red[i][lane], acc[i]);
    __syncthreads();
    for (int i = warp; i < m; i += kSkWarps)
        if (col_ok) C[static_cast<int64_t>(i) * n + j] = red[i][lane];
}

// Any k or alignment: byte loads.
__global__ void __launch_bounds__(kSkWarps * 32) skinny_bytes_kernel(const int8_t* __restrict__ A,
                                                                     const int8_t* __restrict__ Bt,
                                                                     int32_t* __restrict__ C, int m, int64_t n,
                                                                     int64_t k) {
    __shared__ int32_t red[64][kSkCols];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int t = threadIdx.x; t < 64 * kSkCols; t += blockDim.x) (&red[0][0])[t] = 0;
    __syncthreads();
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kSkCols + lane;
    const bool col_ok = j < n;
    for (int i = 0; i < m; ++i) {
        int32_t s = 0;
        if (col_ok)
            for (int64_t kk = warp; kk < k; kk += kSkWarps)
                s += static_cast<int32_t>(A[static_cast<int64_t>(i) * k + kk]) * static_cast<int32_t>(Bt[j * k + kk]);
        atomicAdd(&red[i][lane], s);
    }
    __syncthreads();
    for (int i = warp; i < m; i += kSkWarps)
        if (col_ok) C[static_cast<int64_t>(i) * n + j] = red[i][lane];
}

}  // namespace

cudaError_t launch_skinny_i8(const int8_t* A, const int8_t* Bt, int32_t* C, int64_t m, int64_t n, int64_t k,
                             int num_sms, cudaStream_t stream) {
    (void)num_sms;
    if (m < 1 || m > 128) return cudaErrorInvalidValue;
    if (m > 64) {
        // rows 0..63, then the rest
        const cudaError_t e = launch_skinny_i8(A, Bt, C, 64, n, k, num_sms, stream);
        if (e != cudaSuccess) return e;
        return launch_skinny_i8(A + 64 * k, Bt, C + 64 * n, m - 64, n, k, num_sms, stream);
    }
    const unsigned grid = static_cast<unsigned>((n + kSkCols - 1) / kSkCols);
    const bool vec = (k % 16) == 0 &&
                     ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(Bt)) & 15u) == 0;
    const int mi = static_cast<int>(m);
    if (!vec)
        skinny_bytes_kernel<<<grid, kSkWarps * 32, 0, stream>>>(A, Bt, C, mi, n, k);
    else if (m <= 8)
        skinny_dp4a_kernel<8><<<grid, kSkWarps * 32, 0, stream>>>(A, Bt, C, mi, n, k);
    else if (m <= 16)
        skinny_dp4a_kernel<16><<<grid, kSkWarps * 32, 0, stream>>>(A, Bt, C, mi, n, k);
    else if (m <= 32)
        skinny_dp4a_kernel<32><<<grid, kSkWarps * 32, 0, stream>>>(A, Bt, C, mi, n, k);
    else
        skinny_dp4a_kernel<64><<<grid, kSkWarps * 32, 0, stream>>>(A, Bt, C, mi, n, k);
    return cudaGetLastError();
}

}  // namespace gemm
