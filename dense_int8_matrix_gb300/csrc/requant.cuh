// Requantisation of exact int32 GEMM results, shared by the tensor kernels'
// epilogues and the elementwise requant kernel:
//
//   D[i][j] = q( (float(C[i][j]) * row_scale[i]) * col_scale[j] )
//
// every step one binary32 operation rounded to nearest even (__int2float_rn,
// __fmul_rn: no contraction, no reassociation); q = bfloat16, round to
// nearest even (cvt.rn.bf16x2.f32), or int8: nearest integer with ties to
// even (cvt.rni.s32.f32, which gives 0 for NaN and saturates), clamped to
// [-128, 127].
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace gemm {

__device__ __forceinline__ float rq_value(int32_t c, float rs, float cs) {
    return __fmul_rn(__fmul_rn(__int2float_rn(c), rs), cs);
}

__device__ __forceinline__ uint32_t rq_i8(float z) {
    int v = __float2int_rn(z);
    v = v < -128 ? -128 : (v > 127 ? 127 : v);
    return static_cast<uint32_t>(v) & 0xffu;
}

__device__ __forceinline__ uint32_t rq_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // .x (low half) = lo
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Eight consecutive results t[0..7] of row `row`, columns [c0, c0 + 8), c0 a
// multiple of 8 (so the column scales load as two aligned float4); rs is the
// row's scale.  Rows and columns outside D are skipped.
__device__ __forceinline__ void requant_store8(const RqOut& o, int64_t m, int64_t n, int64_t row, int64_t c0,
                                               float rs, const int32_t (&t)[8]) {
    if (row >= m || c0 >= n) return;
    const bool full = c0 + 8 <= n;
    float cs[8];
    if (full) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(o.col_scale + c0));
        const float4 b = __ldg(reinterpret_cast<const float4*>(o.col_scale + c0) + 1);
        cs[0] = a.x; cs[1] = a.y; cs[2] = a.z; cs[3] = a.w;
        cs[4] = b.x; cs[5] = b.y; cs[6] = b.z; cs[7] = b.w;
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) cs[j] = c0 + j < n ? __ldg(o.col_scale + c0 + j) : 0.f;
    }
    float z[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) z[j] = rq_value(t[j], rs, cs[j]);
    if (o.qmode == kQuantBf16) {
        uint16_t* out = static_cast<uint16_t*>(o.D) + row * o.ldd + c0;
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) w[h] = rq_bf16x2(z[2 * h], z[2 * h + 1]);
        if (full && o.d_vec) {
            *reinterpret_cast<uint4*>(out) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (c0 + j < n) out[j] = static_cast<uint16_t>(w[j >> 1] >> (16 * (j & 1)));
        }
    } else {
        int8_t* out = static_cast<int8_t*>(o.D) + row * o.ldd + c0;
        uint32_t w[2];
#pragma unroll
        for (int h = 0; h < 2; ++h)
            w[h] = rq_i8(z[4 * h]) | (rq_i8(z[4 * h + 1]) << 8) | (rq_i8(z[4 * h + 2]) << 16) |
                   (rq_i8(z[4 * h + 3]) << 24);
        if (full && o.d_vec) {
            *reinterpret_cast<uint2*>(out) = make_uint2(w[0], w[1]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (c0 + j < n) out[j] = static_cast<int8_t>(w[j >> 2] >> (8 * (j & 3)));
        }
    }
}

}  // namespace gemm
