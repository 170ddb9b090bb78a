// Elementwise requantisation of int32 results that no single CTA completes:
// the tiles of a K-split tensor-path launch (each slice adds into int32
// scratch) and the skinny path's C (every CTA adds its K range into it).
// Whole tiles are requantised in the tensor kernels' epilogues instead.
#include <cuda_runtime.h>

#include <cstring>

#include "internal.h"
#include "ptx.cuh"
#include "requant.cuh"

namespace gemm {

namespace {

// One item = eight consecutive columns of one row: all of C (t.bm == 0), or
// the rows of the tiles [tile_from, tile_to) of a bm x bn tiling of C in the
// tensor kernels' tile order.
__global__ void __launch_bounds__(256) requant_kernel(const int32_t* __restrict__ C, int64_t ldc, const RqOut o,
                                                      int64_t m, int64_t n, const RqTiles t) {
    pdl_launch_dependents();
    pdl_wait();   // C is written by the GEMM kernel just before
    const bool all = t.bm == 0;
    const int64_t gpr = all ? (n + 7) / 8 : t.bn / 8;             // 8-column groups per row (of C or a tile)
    const int64_t per_tile = all ? 0 : static_cast<int64_t>(t.bm) * gpr;
    const int64_t items = all ? m * gpr : per_tile * (t.tile_to - t.tile_from);
    const bool c_vec = (ldc & 3) == 0 && (reinterpret_cast<uintptr_t>(C) & 15) == 0;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < items; i += stride) {
        int64_t row, c0;
        if (all) {
            row = i / gpr;
            c0 = (i - row * gpr) * 8;
        } else {
            const int64_t ti = i / per_tile;
            const int64_t local = i - ti * per_tile;
            int tm, tn;
            tc_tile_coords(static_cast<int>(t.tile_from + ti), t.tiles_m, t.tiles_n, tm, tn);
            const int64_t r = local / gpr;
            row = static_cast<int64_t>(tm) * t.bm + r;
            c0 = static_cast<int64_t>(tn) * t.bn + (local - r * gpr) * 8;
        }
        if (row >= m || c0 >= n) continue;
        const int32_t* src = C + row * ldc + c0;
        int32_t v[8];
        if (c_vec && c0 + 8 <= n) {
            const int4 a = __ldg(reinterpret_cast<const int4*>(src));
            const int4 b = __ldg(reinterpret_cast<const int4*>(src) + 1);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = c0 + j < n ? src[j] : 0;
        }
        requant_store8(o, m, n, row, c0, __ldg(o.row_scale + row), v);
    }
}

}  // namespace

cudaError_t launch_requant(const int32_t* C, int64_t ldc, const RqOut& o, int64_t m, int64_t n, const RqTiles& t,
                           int num_sms, cudaStream_t stream) {
    const int64_t gpr = t.bm == 0 ? (n + 7) / 8 : t.bn / 8;
    const int64_t items = t.bm == 0 ? m * gpr : static_cast<int64_t>(t.bm) * gpr * (t.tile_to - t.tile_from);
    if (items <= 0) return cudaSuccess;
    int64_t grid = (items + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (grid > cap) grid = cap;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, requant_kernel, C, ldc, o, m, n, t);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace gemm
