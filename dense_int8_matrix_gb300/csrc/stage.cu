// Operand staging for the tensor-core path.
//
// sm_103a has no integer tensor-core MMA (ptxas rejects tcgen05.mma
// .kind::i8 for this target), so int8 operands are widened to f16, in which
// every int8 value is exact, and multiplied on the f16 tensor cores.  The
// same pass re-pitches rows whose length is not a multiple of 16 bytes, which
// TMA requires of every row pitch; the pad is never read (the tensor map's K
// extent is k, so TMA fills K beyond it with zeros).
//
// int8 -> f16 without a conversion instruction: for a byte x, the f16 bit
// pattern 0x6400 | (x ^ 0x80) encodes 1024 + (x + 128); subtracting 1152 (exact
// in f16) leaves x.  Memory-bound: 1 byte read and 2 written per element.
//
// Large contiguous operands go through shared memory with bulk copies
// (cp.async.bulk): 8 KiB int8 chunks in (four in flight), widened in shared
// memory, 16 KiB f16 chunks out, three 66 KiB CTAs per SM.  Measured on GB300
// for the 4096^3 operands (32 MiB in, 64 MiB out) inside the GEMM step: 20.4
// us per launch, against 24.8 us with one CTA per SM (16 KiB chunks, four or
// up to ten in flight: 23.1-24.8 us) -- a CTA converts a chunk between two
// barriers, so more CTAs, not more loads in flight, keep HBM busy; 4 KiB
// chunks at six CTAs per SM measured the same (19.9 us).  Per-thread 16-byte
// loads and stores took 24.8 us.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace gemm {

namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void convert16(const uint4 v, uint4* d) {
    const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
    uint4 lo, hi;
    lo.x = i8x2_to_f16x2(w[0], 0x4140u);
    lo.y = i8x2_to_f16x2(w[0], 0x4342u);
    lo.z = i8x2_to_f16x2(w[1], 0x4140u);
    lo.w = i8x2_to_f16x2(w[1], 0x4342u);
    hi.x = i8x2_to_f16x2(w[2], 0x4140u);
    hi.y = i8x2_to_f16x2(w[2], 0x4342u);
    hi.z = i8x2_to_f16x2(w[3], 0x4140u);
    hi.w = i8x2_to_f16x2(w[3], 0x4342u);
    d[0] = lo;
    d[1] = hi;
}

constexpr int kStageUnroll = 4;

// Items of the zeroing work: 4 consecutive words of C (of all of C, or of a
// row of a split tile), so that consecutive threads write consecutive 16-byte
// pieces.
__host__ __device__ inline int64_t zero_items(const StageZero& z) {
    if (z.C == nullptr) return 0;
    if (z.bm == 0) return (z.m * z.n + 3) / 4;
    return static_cast<int64_t>(z.tile_to - z.tile_from) * z.bm * (z.bn / 4);
}

__device__ __forceinline__ void zero4(int32_t* p, int64_t avail, bool vec) {
    if (vec && avail >= 4)
        *reinterpret_cast<uint4*>(p) = make_uint4(0u, 0u, 0u, 0u);
    else
        for (int64_t j = 0; j < 4 && j < avail; ++j) p[j] = 0;
}

__device__ __forceinline__ void zero_work(const StageZero& z, int64_t i0, int64_t stride) {
    const int64_t items = zero_items(z);
    const bool vec = (z.n % 4) == 0 && (reinterpret_cast<uintptr_t>(z.C) & 15u) == 0;
    if (z.bm == 0) {
        const int64_t total = z.m * z.n;
        for (int64_t i = i0; i < items; i += stride) zero4(z.C + 4 * i, total - 4 * i, vec);
        return;
    }
    const int64_t q4 = z.bn / 4, per_tile = static_cast<int64_t>(z.bm) * q4;
    for (int64_t i = i0; i < items; i += stride) {
        const int t = z.tile_from + static_cast<int>(i / per_tile);
        const int64_t rem = i % per_tile;
        const int r = static_cast<int>(rem / q4);
        const int64_t c = 4 * (rem % q4);
        int tm, tn;
        tc_tile_coords(t, z.tiles_m, z.tiles_n, tm, tn);
        const int64_t row = static_cast<int64_t>(tm) * z.bm + r;
        const int64_t col = static_cast<int64_t>(tn) * z.bn + c;
        if (row < z.m && col < z.n) zero4(z.C + row * z.n + col, z.n - col, vec);
    }
}

// ---- bulk-copy staging -------------------------------------------------
constexpr int kBulkChunk = 8192;                   // int8 bytes per chunk
constexpr int kBulkDepth = 4;                      // chunks in flight per CTA
constexpr int kBulkThreads = 256;
constexpr size_t kBulkSmem = static_cast<size_t>(kBulkDepth) * kBulkChunk + 2 * 2 * kBulkChunk + 1024;
constexpr int64_t kBulkMinBytes = int64_t(8) << 20;   // smaller problems: per-thread kernel
constexpr int kBulkCtasPerSm = 3;
static_assert(kBulkCtasPerSm * (kBulkSmem + 1024) <= 233472, "bulk staging CTAs per SM");

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Chunk c of the concatenated A | Bt bytes: source, destination, length.
struct BulkChunk {
    const uint8_t* src;
    uint8_t* dst;
    uint32_t len;
};

__device__ __forceinline__ BulkChunk bulk_chunk(int64_t c, const uint8_t* A, const uint8_t* Bt, uint8_t* Ah,
                                                uint8_t* Bh, int64_t a_bytes, int64_t b_bytes, int64_t na) {
    BulkChunk x;
    const bool isA = c < na;
    const int64_t off = (isA ? c : c - na) * kBulkChunk;
    const int64_t total = isA ? a_bytes : b_bytes;
    x.src = (isA ? A : Bt) + off;
    x.dst = (isA ? Ah : Bh) + 2 * off;
    x.len = static_cast<uint32_t>(total - off < kBulkChunk ? total - off : kBulkChunk);
    return x;
}

// Contiguous rows (k == k_pitch, k % 16 == 0, 16-byte aligned): chunks of A
// then of Bt, grid-stride over CTAs; every wait bounded.
__global__ void __launch_bounds__(kBulkThreads) stage_i8_bulk_kernel(const uint8_t* __restrict__ A,
                                                                     const uint8_t* __restrict__ Bt,
                                                                     uint8_t* __restrict__ Ah, uint8_t* __restrict__ Bh,
                                                                     int64_t a_bytes, int64_t b_bytes,
                                                                     const StageZero z, int* err) {
    pdl_launch_dependents();   // the GEMM kernel after this one may start its set-up
    pdl_wait();                // launched ahead of the kernel before: touch nothing until it completes
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sin = base;                                 // kBulkDepth x 8 KiB
    const uint32_t sout = base + kBulkDepth * kBulkChunk;      // 2 x 16 KiB
    uint8_t* const gin = smem_raw + (base - smem_u32(smem_raw));
    uint8_t* const gout = gin + kBulkDepth * kBulkChunk;
    __shared__ __align__(8) uint64_t full[kBulkDepth];
    __shared__ uint32_t abort_flag;

    zero_work(z, static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x, static_cast<int64_t>(gridDim.x) * blockDim.x);

    const int64_t na = (a_bytes + kBulkChunk - 1) / kBulkChunk;
    const int64_t nchunks = na + (b_bytes + kBulkChunk - 1) / kBulkChunk;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kBulkDepth; ++s) mbar_init(smem_u32(&full[s]), 1);
        abort_flag = 0u;
        fence_barrier_init();
    }
    __syncthreads();
    const int64_t step = gridDim.x;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kBulkDepth; ++s) {
            const int64_t c = blockIdx.x + s * step;
            if (c >= nchunks) break;
            const BulkChunk x = bulk_chunk(c, A, Bt, Ah, Bh, a_bytes, b_bytes, na);
            mbar_arrive_expect_tx(smem_u32(&full[s]), x.len);
            bulk_load(sin + s * kBulkChunk, x.src, x.len, smem_u32(&full[s]));
        }
    }
    uint32_t it = 0;
    for (int64_t c = blockIdx.x; c < nchunks; c += step, ++it) {
        const uint32_t s = it % kBulkDepth, ph = (it / kBulkDepth) & 1u;
        const BulkChunk x = bulk_chunk(c, A, Bt, Ah, Bh, a_bytes, b_bytes, na);
        int got = 1;
        if (threadIdx.x == 0) {
            got = wait_bounded(smem_u32(&full[s]), ph, &abort_flag, err, kDevErrTimeoutProducer) ? 1 : 0;
            bulk_wait_read_1();   // the output buffer stored two chunks ago has been read
        }
        got = __syncthreads_and(got);
        if (!got) break;
        const uint4* in = reinterpret_cast<const uint4*>(gin + s * kBulkChunk);
        uint4* out = reinterpret_cast<uint4*>(gout + (it & 1u) * 2 * kBulkChunk);
        for (uint32_t i = threadIdx.x; i < x.len / 16; i += blockDim.x) convert16(in[i], out + 2 * i);
        fence_proxy_async_smem();   // the bulk store (async proxy) reads what the threads wrote
        __syncthreads();
        if (threadIdx.x == 0) {
            bulk_store(x.dst, sout + (it & 1u) * 2 * kBulkChunk, 2 * x.len);
            bulk_commit();
            const int64_t cn = c + kBulkDepth * step;   // refill the slot just read
            if (cn < nchunks) {
                const BulkChunk y = bulk_chunk(cn, A, Bt, Ah, Bh, a_bytes, b_bytes, na);
                mbar_arrive_expect_tx(smem_u32(&full[s]), y.len);
                bulk_load(sin + s * kBulkChunk, y.src, y.len, smem_u32(&full[s]));
            }
        }
    }
    if (threadIdx.x == 0) {
        bulk_wait_all();
        // loads still in flight after an early exit must land before the CTA ends
        for (uint32_t j = 0; j < kBulkDepth; ++j) {
            const uint32_t n = it + j;   // slots of the next kBulkDepth chunks
            const int64_t c = blockIdx.x + static_cast<int64_t>(n) * step;
            if (c >= nchunks) break;
            wait_bounded(smem_u32(&full[n % kBulkDepth]), (n / kBulkDepth) & 1u, nullptr, err, kDevErrTimeoutTeardown);
        }
    }
    __syncthreads();
}

// Contiguous rows (k == k_pitch, k % 16 == 0): 16 int8 -> 16 f16 per item;
// each thread keeps kStageUnroll loads in flight.
__global__ void __launch_bounds__(256) stage_i8_flat_kernel(const uint4* __restrict__ srcA,
                                                            const uint4* __restrict__ srcB, uint4* __restrict__ dstA,
                                                            uint4* __restrict__ dstB, int64_t itemsA,
                                                            int64_t itemsB, const StageZero z) {
    pdl_launch_dependents();   // the GEMM kernel after this one may start its set-up
    pdl_wait();                // launched ahead of the kernel before: touch nothing until it completes
    const int64_t total = itemsA + itemsB;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    zero_work(z, static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x, stride);
    for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < total;
         i0 += stride * kStageUnroll) {
        uint4 v[kStageUnroll];
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < total) v[u] = ld_stream(i < itemsA ? srcA + i : srcB + (i - itemsA));
        }
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < total) convert16(v[u], i < itemsA ? dstA + 2 * i : dstB + 2 * (i - itemsA));
        }
    }
}

// Any k or alignment: rows re-pitched to k_pitch (a multiple of 8); each item
// is 8 elements of a row (byte loads, zero beyond k) and one 16-byte store.
__global__ void __launch_bounds__(256) stage_i8_rows_kernel(const int8_t* __restrict__ A,
                                                            const int8_t* __restrict__ Bt, uint4* __restrict__ Ah,
                                                            uint4* __restrict__ Bh, int64_t m, int64_t n, int64_t k,
                                                            int64_t k_pitch, const StageZero z) {
    pdl_launch_dependents();   // the GEMM kernel after this one may start its set-up
    pdl_wait();                // launched ahead of the kernel before: touch nothing until it completes
    const int64_t cpr = k_pitch / 8;   // 8-element pieces per staged row
    const int64_t itemsA = m * cpr;
    const int64_t total = itemsA + n * cpr;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    zero_work(z, static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x, stride);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const bool isA = i < itemsA;
        const int64_t j = isA ? i : i - itemsA;
        const int64_t row = j / cpr, c = j - row * cpr;
        const uint8_t* src = reinterpret_cast<const uint8_t*>(isA ? A : Bt) + row * k + c * 8;
        const int64_t left = k - c * 8;
        uint32_t w[2] = {0u, 0u};   // zero bytes widen to 0 (the pad beyond k)
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (e < left) w[e >> 2] |= static_cast<uint32_t>(src[e]) << (8 * (e & 3));
        const uint32_t w0 = w[0] ^ 0x80808080u, w1 = w[1] ^ 0x80808080u;
        (isA ? Ah : Bh)[row * cpr + c] = make_uint4(i8x2_to_f16x2(w0, 0x4140u), i8x2_to_f16x2(w0, 0x4342u),
                                                    i8x2_to_f16x2(w1, 0x4140u), i8x2_to_f16x2(w1, 0x4342u));
    }
}

// 16-bit copy with re-pitched rows: 8 elements per item (2-byte loads, zero
// beyond k), one 16-byte store.
__global__ void __launch_bounds__(256) stage_b16_rows_kernel(const uint16_t* __restrict__ A,
                                                             const uint16_t* __restrict__ Bt,
                                                             uint4* __restrict__ Ah, uint4* __restrict__ Bh,
                                                             int64_t m, int64_t n, int64_t k, int64_t k_pitch) {
    pdl_launch_dependents();   // the GEMM kernel after this one may start its set-up
    pdl_wait();                // launched ahead of the kernel before: touch nothing until it completes
    const int64_t cpr = k_pitch / 8;
    const int64_t itemsA = m * cpr;
    const int64_t total = itemsA + n * cpr;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const bool isA = i < itemsA;
        const int64_t j = isA ? i : i - itemsA;
        const int64_t row = j / cpr, c = j - row * cpr;
        const uint16_t* src = (isA ? A : Bt) + row * k + c * 8;
        const int64_t left = k - c * 8;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (e < left) w[e >> 1] |= static_cast<uint32_t>(src[e]) << (16 * (e & 1));
        (isA ? Ah : Bh)[row * cpr + c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Skinny-path prologue: A to f16 and all of C zeroed.  128 threads at <= 32
// registers (4,096 registers) and no shared memory fit on an SM beside a
// running skinny tensor-core CTA (640 threads x 96 registers, <= 226 KiB of
// shared memory), so with programmatic stream serialization every CTA of this
// kernel is resident, and has let the skinny kernel behind it launch, while
// the kernel before it still runs; the skinny CTAs then take each SM as soon
// as it is free and stream their Bt into L2 while this kernel waits.  Nothing
// is read or written before the wait: A, A16 and C may all be in use by the
// kernel before.
constexpr int kProThreads = 128;
__global__ void __launch_bounds__(kProThreads, 16) skinny_prologue_kernel(const uint4* __restrict__ A,
                                                                          uint4* __restrict__ A16, int64_t itemsA,
                                                                          const StageZero z) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int64_t i0 = t; i0 < itemsA; i0 += 2 * stride) {
        uint4 v[2];
#pragma unroll
        for (int u = 0; u < 2; ++u)
            if (i0 + u * stride < itemsA) v[u] = ld_stream(A + i0 + u * stride);
#pragma unroll
        for (int u = 0; u < 2; ++u)
            if (i0 + u * stride < itemsA) convert16(v[u], A16 + 2 * (i0 + u * stride));
    }
    zero_work(z, t, stride);
}

// Launch with programmatic stream serialization: the kernel may become
// resident while the kernel before it in the stream still runs (if that one
// lets its dependents start early); every staging kernel waits for it
// (pdl_wait) before touching memory.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kern)(Params...), int grid, int block, size_t smem, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(block), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Params>(args)...);
}

int grid_for(int64_t items, int num_sms) {
    // 8 resident 256-thread blocks per SM, grid a multiple of the SM count
    int64_t want = (items + 255) / 256;
    int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (want > cap) want = cap;
    if (want < 1) want = 1;
    return static_cast<int>(want);
}

}  // namespace

cudaError_t launch_stage_i8(const int8_t* A, const int8_t* Bt, uint16_t* Ah, uint16_t* Bh, int64_t m, int64_t n,
                            int64_t k, int64_t k_pitch, const StageZero& z, int* err, int num_sms,
                            cudaStream_t stream) {
    const bool aligned = ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(Bt) |
                           reinterpret_cast<uintptr_t>(Ah) | reinterpret_cast<uintptr_t>(Bh)) &
                          15u) == 0;
    if (k == k_pitch && (k % 16) == 0 && aligned && (m + n) * k >= kBulkMinBytes && err != nullptr) {
        cudaError_t e = kernel_attrs_once(reinterpret_cast<const void*>(stage_i8_bulk_kernel),
                                          static_cast<int>(kBulkSmem), false);
        if (e != cudaSuccess) return e;
        const int64_t chunks = ((m * k + kBulkChunk - 1) / kBulkChunk) + ((n * k + kBulkChunk - 1) / kBulkChunk);
        // three CTAs per SM (66 KiB of shared memory each)
        const int64_t cap = static_cast<int64_t>(kBulkCtasPerSm) * num_sms;
        const int grid = static_cast<int>(chunks < cap ? chunks : cap);
        e = launch_pdl(stage_i8_bulk_kernel, grid, kBulkThreads, kBulkSmem, stream,
                       reinterpret_cast<const uint8_t*>(A), reinterpret_cast<const uint8_t*>(Bt),
                       reinterpret_cast<uint8_t*>(Ah), reinterpret_cast<uint8_t*>(Bh), m * k, n * k, z, err);
        if (e != cudaSuccess) return e;
    } else if (k == k_pitch && (k % 16) == 0 && aligned) {
        const int64_t itemsA = m * k / 16, itemsB = n * k / 16;
        const int64_t zi = zero_items(z);
        const int64_t work = itemsA + itemsB > zi ? itemsA + itemsB : zi;
        cudaError_t e = launch_pdl(stage_i8_flat_kernel, grid_for(work, num_sms), 256, 0, stream,
                                   reinterpret_cast<const uint4*>(A), reinterpret_cast<const uint4*>(Bt),
                                   reinterpret_cast<uint4*>(Ah), reinterpret_cast<uint4*>(Bh), itemsA, itemsB, z);
        if (e != cudaSuccess) return e;
    } else {
        const int64_t items = (m + n) * (k_pitch / 8);
        const int64_t zi = zero_items(z);
        cudaError_t e = launch_pdl(stage_i8_rows_kernel, grid_for(items > zi ? items : zi, num_sms), 256, 0, stream,
                                   A, Bt, reinterpret_cast<uint4*>(Ah), reinterpret_cast<uint4*>(Bh), m, n, k,
                                   k_pitch, z);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_skinny_prologue(const int8_t* A, uint16_t* A16, int32_t* C, int64_t m, int64_t n, int64_t k,
                                   int num_sms, cudaStream_t stream) {
    StageZero z;   // all of C
    z.C = C;
    z.m = m;
    z.n = n;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms), 1, 1);
    cfg.blockDim = dim3(kProThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, skinny_prologue_kernel, reinterpret_cast<const uint4*>(A),
                                       reinterpret_cast<uint4*>(A16), m * k / 16, z);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_stage_b16(const uint16_t* A, const uint16_t* Bt, uint16_t* Ah, uint16_t* Bh, int64_t m,
                             int64_t n, int64_t k, int64_t k_pitch, int num_sms, cudaStream_t stream) {
    cudaError_t e = launch_pdl(stage_b16_rows_kernel, grid_for((m + n) * (k_pitch / 8), num_sms), 256, 0, stream, A,
                               Bt, reinterpret_cast<uint4*>(Ah), reinterpret_cast<uint4*>(Bh), m, n, k, k_pitch);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace gemm
