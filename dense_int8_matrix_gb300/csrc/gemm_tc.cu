// Tensor-core GEMM for sm_103a: C = A x B with A (m x k) and B stored K-major
// as Bt (n x k), both staged as 16-bit operands (f16 holding exact int8
// values, or bf16), fp32 accumulation in TMEM, int32 or fp32 output.
//
// Structure (one persistent CTA per SM slot, 12 warps):
//   warp 0      TMA producer: copies the A tile (BM x 64) and the Bt tile
//               (BN x 64) of each K step into a 4-stage shared-memory ring
//               (128-byte swizzle), signalling a "full" mbarrier per stage.
//               This multi-stage ring is the double-buffered prefetch of
//               "CUDA编程实践" §3 (数据prefetch) taken to four stages.
//   warp 1      allocates TMEM and issues tcgen05.mma (M = BM, N = BN, K = 16,
//               four per stage) into one of two TMEM accumulators; each
//               stage is released to the producer by tcgen05.commit.
//   warps 4-11  epilogue: tcgen05.ld the accumulator, fold it into running
//               sums held in registers, release the accumulator, and after
//               the last K chunk of a tile write C with vector stores.
// The two accumulators alternate per K chunk, so the epilogue of one chunk
// (or tile) overlaps the MMAs of the next.
//
// For int8 problems the accumulator is drained every 1024 K elements and
// converted to int32 exactly (see kI8ChunkK), so the result is bit-exact for
// every int8 input up to the library's k limit.  For bf16 problems a chunk is
// the whole K loop.
//
// Tile order: tiles are visited in bands of 8 M-tiles, N fastest within a
// band, so that the CTAs running together share A and B panels in L2 (the
// swizzled block mapping of "先导杯比赛回顾", section "Swizzle 线程块映射").
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "requant.cuh"

namespace gemm {

namespace {

template <int BM, int BN>
struct TcCfg {
    static constexpr int A_BYTES = BM * kTcRowBytes;
    static constexpr int B_BYTES = BN * kTcRowBytes;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = tc_tmem_cols(BN);
    static constexpr int HALF = BN / 2;                 // columns per epilogue thread
    static constexpr int SLICE = HALF >= 32 ? 32 : 16;  // columns per tcgen05.ld
    static constexpr int NSLICE = HALF / SLICE;
    static constexpr bool TMA_STORE = tc_tma_store_tile(BM, BN);
    static constexpr int EPI_BYTES = TMA_STORE ? kTcEpilogueWarps * kTcEpiStageBytes : 0;
    static constexpr size_t SMEM = tc_smem_bytes(BM, BN);
    static_assert(BM == 64 || BM == 128, "BM");
    static_assert(BN == 32 || BN == 64 || BN == 128 || BN == 256, "BN");
    static_assert(kTcStages * STAGE_BYTES + EPI_BYTES + 1024 + 8 * (2 * kTcStages + 5) + 8 <= SMEM, "smem layout");
};

struct TcParams {
    void* C;
    int* err;
    int c_tma;      // 1: write C with TMA stores (wide tiles, n % 4 == 0, C 16-byte aligned)
    int64_t m, n;
    int64_t ldc;    // row pitch of C in elements
    int num_kb;     // ceil(k / 64)
    int chunk_kb;   // K steps per accumulator chunk
    int tiles_m, tiles_n, tiles;
    RqOut rq;       // qmode != none: whole tiles requantised into rq.D, not written to C
    int units;      // split_from + (tiles - split_from) * split_k
    int split_from; // tiles [split_from, tiles) run as split_k K slices each (C zeroed over them)
    int split_k;
};

// A unit of work: one tile over the K steps [kb_lo, kb_hi).  Units below
// split_from are whole tiles; above it, the slices of a split tile are
// consecutive units (so they run in the same round on different CTAs), each
// a run of whole K steps.
struct Unit {
    int tm, tn, kb_lo, kb_hi;
    int split_tile;   // index among the split tiles, -1 if the tile is whole
    int slice;
};

__device__ __forceinline__ Unit unit_at(int u, const TcParams& p) {
    Unit x;
    int t;
    if (u < p.split_from) {
        t = u;
        x.kb_lo = 0;
        x.kb_hi = p.num_kb;
        x.split_tile = -1;
        x.slice = 0;
    } else {
        const int v = u - p.split_from;
        x.split_tile = v / p.split_k;
        x.slice = v - x.split_tile * p.split_k;
        t = p.split_from + x.split_tile;
        // K steps [kb_lo, kb_hi): accumulated in chunks of chunk_kb steps
        // from kb_lo, so every fp32 chunk stays exact
        x.kb_lo = x.slice * p.num_kb / p.split_k;
        x.kb_hi = (x.slice + 1) * p.num_kb / p.split_k;
    }
    tc_tile_coords(t, p.tiles_m, p.tiles_n, x.tm, x.tn);
    return x;
}

template <int BM, int BN, bool INT_OUT, bool C_TMA>
__global__ void __launch_bounds__(kTcThreads, (BN >= 128 ? 1 : 2))
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcParams p) {
    using Cfg = TcCfg<BM, BN>;
    extern __shared__ uint8_t smem_raw[];

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sA = base;
    const uint32_t sB = base + kTcStages * Cfg::A_BYTES;
    const uint32_t sEpi = base + kTcStages * Cfg::STAGE_BYTES;   // 8 x 4 KiB, 1024-aligned
    uint8_t* ctrl = smem_raw + (base - raw) + kTcStages * Cfg::STAGE_BYTES + Cfg::EPI_BYTES;
    const uint32_t bar0 = smem_u32(ctrl);
    // barrier slots: full[S], empty[S], acc_full[2], acc_empty[2], done
    const uint32_t full_bar0 = bar0;
    const uint32_t empty_bar0 = bar0 + 8u * kTcStages;
    const uint32_t accf_bar0 = bar0 + 16u * kTcStages;
    const uint32_t acce_bar0 = accf_bar0 + 16u;
    const uint32_t done_bar = acce_bar0 + 16u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 8 * (2 * kTcStages + 5));
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5;
    // the next kernel in the stream (the next call's staging kernel, which
    // waits for this one before it touches memory) may launch
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(full_bar0 + 8u * s, 1);
            mbar_init(empty_bar0 + 8u * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar0 + 8u * b, 1);
            mbar_init(acce_bar0 + 8u * b, kTcEpilogueWarps);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0u;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the epilogue writes C (zeroed over the split tiles by the staging
    // kernel) only after the kernel before this one in the stream
    // (programmatic dependent launch)
    if (warp >= 4) {
        pdl_wait();
        fence_proxy_async_global();   // TMA reduce-adds below follow the zeroing
    }

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer --
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            if (C_TMA) tma_prefetch_desc(&tmC);
            pdl_wait();   // the operands may come from the staging kernel just before
            const uint64_t pol = policy_evict_normal();
            uint32_t issued = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
                const Unit w = unit_at(u, p);
                const int tm = w.tm, tn = w.tn;
                for (int kb = w.kb_lo; kb < w.kb_hi; ++kb) {
                    const uint32_t s = issued % kTcStages;
                    const uint32_t ph = (issued / kTcStages) & 1u;
                    if (!wait_bounded(empty_bar0 + 8u * s, ph ^ 1u, abort_flag, p.err, kDevErrTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar0 + 8u * s, Cfg::STAGE_BYTES);
                    tma_load_2d(sA + s * Cfg::A_BYTES, &tmA, kb * kTcBK, tm * BM, full_bar0 + 8u * s, pol);
                    tma_load_2d(sB + s * Cfg::B_BYTES, &tmB, kb * kTcBK, tn * BN, full_bar0 + 8u * s, pol);
                    ++issued;
                }
            }
            // Teardown: every copy started must land before the CTA exits.
            for (uint32_t s = 0; s < static_cast<uint32_t>(kTcStages) && s < issued; ++s) {
                const uint32_t last = s + ((issued - 1u - s) / kTcStages) * kTcStages;
                wait_bounded(full_bar0 + 8u * s, (last / kTcStages) & 1u, nullptr, p.err, kDevErrTimeoutTeardown);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer --
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(INT_OUT ? 0u : 1u, BM, BN);
            uint32_t consumed = 0, acc_iter = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
                const Unit w = unit_at(u, p);
                for (int c0 = w.kb_lo; ok && c0 < w.kb_hi; c0 += p.chunk_kb) {
                    const uint32_t buf = acc_iter & 1u;
                    const uint32_t aph = (acc_iter >> 1) & 1u;
                    if (!wait_bounded(acce_bar0 + 8u * buf, aph ^ 1u, abort_flag, p.err, kDevErrTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * BN;
                    const int c1 = min(w.kb_hi, c0 + p.chunk_kb);
                    for (int kb = c0; kb < c1; ++kb) {
                        const uint32_t s = consumed % kTcStages;
                        const uint32_t ph = (consumed / kTcStages) & 1u;
                        if (!wait_bounded(full_bar0 + 8u * s, ph, abort_flag, p.err, kDevErrTimeoutMma)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t adesc = smem_desc_sw128_kmajor(sA + s * Cfg::A_BYTES);
                        const uint64_t bdesc = smem_desc_sw128_kmajor(sB + s * Cfg::B_BYTES);
#pragma unroll
                        for (int kk = 0; kk < kTcBK / 16; ++kk) {
                            // K step of 16 elements = 32 bytes = 2 in the >>4 address field
                            mma_f16_ss(d_tmem, adesc + 2u * kk, bdesc + 2u * kk, idesc,
                                       (kb > c0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit(empty_bar0 + 8u * s);
                        ++consumed;
                    }
                    if (!ok) break;
                    mma_commit(accf_bar0 + 8u * buf);
                    ++acc_iter;
                }
            }
            // Teardown: all MMAs issued must complete before TMEM is freed.
            mma_commit(done_bar);
            wait_bounded(done_bar, 0u, nullptr, p.err, kDevErrTimeoutTeardown);
        }
    } else if (warp >= 4) {
        // -------------------------------------------------------- epilogue --
        const int e = warp - 4;
        const int q = warp & 3;     // TMEM lane quarter this warp can access
        const int h = e >> 2;       // which half of the BN columns
        uint32_t acc_iter = 0;
        bool ok = true;
        const bool row_valid = (BM == 128) || (lane < 16);
        const int row_in_tile = (BM == 128) ? (q * 32 + lane) : (q * 16 + lane);
        const bool c_vec = ((p.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0);
        for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
            const Unit w = unit_at(u, p);
            const int tm = w.tm, tn = w.tn;
            // every slice of a split tile adds into C (zero over the tile)
            const bool add_into = w.split_tile >= 0;
            const int64_t row = static_cast<int64_t>(tm) * BM + row_in_tile;
            const int64_t col0 = static_cast<int64_t>(tn) * BN + h * Cfg::HALF;
            // int8 problems: exact int32 running sums over the K chunks; bf16
            // problems have a single chunk and need none
            int32_t acc[INT_OUT ? Cfg::HALF : 1];
#pragma unroll
            for (int j = 0; j < (INT_OUT ? Cfg::HALF : 1); ++j) acc[j] = 0;
            for (int c0 = w.kb_lo; c0 < w.kb_hi; c0 += p.chunk_kb) {
                const uint32_t buf = acc_iter & 1u;
                const uint32_t aph = (acc_iter >> 1) & 1u;
                const bool last = c0 + p.chunk_kb >= w.kb_hi;
                // lane 0 polls; the warp then reconverges before the
                // warp-collective tcgen05.ld
                int got = 1;
                if (lane == 0)
                    got = wait_bounded(accf_bar0 + 8u * buf, aph, abort_flag, p.err, kDevErrTimeoutEpilogue) ? 1 : 0;
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tcol = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * BN + h * Cfg::HALF;
#pragma unroll
                for (int sl = 0; sl < Cfg::NSLICE; ++sl) {
                    uint32_t r[INT_OUT ? 1 : Cfg::SLICE];
                    if constexpr (INT_OUT) {
                        // 16 columns at a time keeps the registers live beside the
                        // running sums low
#pragma unroll
                        for (int half = 0; half < Cfg::SLICE / 16; ++half) {
                            uint32_t v[16];
                            tmem_ld_32x32b_x16(tcol + sl * Cfg::SLICE + half * 16, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                // exact: an fp32 chunk sum is an integer of magnitude <= 2^24
                                acc[sl * Cfg::SLICE + half * 16 + j] += __float2int_rn(__uint_as_float(v[j]));
                            }
                        }
                    } else {
                        if constexpr (Cfg::SLICE == 32)
                            tmem_ld_32x32b_x32(tcol + sl * 32, r);
                        else
                            tmem_ld_32x32b_x16(tcol + sl * 16, r);
                        tmem_wait_ld();
                    }
                    if (!last) continue;
                    // this slice's final 32-bit results: the int32 sums, or the
                    // fp32 values as loaded
#define GEMM_TC_OUT(j) (INT_OUT ? static_cast<uint32_t>(acc[(INT_OUT ? sl * Cfg::SLICE : 0) + (j)]) : r[INT_OUT ? 0 : (j)])
                    const int64_t cs = col0 + sl * Cfg::SLICE;
                    if constexpr (INT_OUT) {
                        if (p.rq.qmode != kQuantNone && !add_into) {
                            // a whole tile: its exact sums are final, requantise
                            // them straight into D (eight columns per store)
                            if (row_valid) {
                                const float rs = row < p.m ? __ldg(p.rq.row_scale + row) : 0.f;
#pragma unroll
                                for (int g = 0; g < Cfg::SLICE / 8; ++g) {
                                    int32_t t[8];
#pragma unroll
                                    for (int j = 0; j < 8; ++j) t[j] = acc[sl * Cfg::SLICE + g * 8 + j];
                                    requant_store8(p.rq, p.m, p.n, row, cs + g * 8, rs, t);
                                }
                            }
                            continue;
                        }
                    }
                    if constexpr (C_TMA) {
                        // Coalesced write-back (the shared-memory staged epilogue of
                        // "先导杯比赛回顾", section "Epilogue 写回优化"): each lane writes
                        // its row of the 32-column slice (128 bytes) into the warp's
                        // 128B-swizzled 4 KiB buffer, then one TMA store moves the
                        // 32 x 32 box to C; rows / columns outside C are clipped.
                        static_assert(!C_TMA || Cfg::SLICE == 32, "TMA store slices are 32 columns");
                        const uint32_t stg = sEpi + e * kTcEpiStageBytes;
                        const uint32_t row_base = stg + lane * 128;
                        if (lane == 0) bulk_wait_read_all();   // the previous box has left the buffer
                        __syncwarp();
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            st_shared_v4(row_base + ((c ^ (lane & 7)) << 4), GEMM_TC_OUT(4 * c), GEMM_TC_OUT(4 * c + 1),
                                         GEMM_TC_OUT(4 * c + 2), GEMM_TC_OUT(4 * c + 3));
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            const int32_t ys = static_cast<int32_t>(static_cast<int64_t>(tm) * BM + q * 32);
                            if (add_into)
                                tma_reduce_add_2d(&tmC, stg, static_cast<int32_t>(cs), ys);
                            else
                                tma_store_2d(&tmC, stg, static_cast<int32_t>(cs), ys);
                            bulk_commit();
                        }
                    } else if constexpr (Cfg::TMA_STORE) {
                        // C that TMA cannot store (unaligned rows or base): the
                        // 32 x 32 block goes through the warp's staging buffer so
                        // that every store (or atomic add) instruction covers 32
                        // consecutive columns of one row
                        const uint32_t stg = sEpi + e * kTcEpiStageBytes;
                        uint32_t vals[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) vals[j] = GEMM_TC_OUT(j);
                        __syncwarp();   // the previous block has been read out
                        stage_rows32(stg, lane, vals);
                        __syncwarp();
                        const int64_t col = cs + lane;
                        const int64_t ytop = static_cast<int64_t>(tm) * BM + q * 32;
#pragma unroll 4
                        for (int j = 0; j < 32; ++j) {
                            const uint32_t v = staged_at(stg, j, lane);
                            if (ytop + j < p.m && col < p.n) {
                                uint32_t* o = static_cast<uint32_t*>(p.C) + (ytop + j) * p.ldc + col;
                                if (add_into)
                                    atomicAdd(o, v);
                                else
                                    *o = v;
                            }
                        }
                    } else {
                        if (row_valid && row < p.m) {
                            uint32_t* out = static_cast<uint32_t*>(p.C) + row * p.ldc + cs;
                            if (add_into) {
#pragma unroll
                                for (int j = 0; j < Cfg::SLICE; ++j)
                                    if (cs + j < p.n) atomicAdd(out + j, GEMM_TC_OUT(j));
                            } else if (c_vec && cs + Cfg::SLICE <= p.n) {
#pragma unroll
                                for (int j = 0; j < Cfg::SLICE; j += 4)
                                    *reinterpret_cast<uint4*>(out + j) =
                                        make_uint4(GEMM_TC_OUT(j), GEMM_TC_OUT(j + 1), GEMM_TC_OUT(j + 2), GEMM_TC_OUT(j + 3));
                            } else {
#pragma unroll
                                for (int j = 0; j < Cfg::SLICE; ++j)
                                    if (cs + j < p.n) out[j] = GEMM_TC_OUT(j);
                            }
                        }
                    }
#undef GEMM_TC_OUT
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce_bar0 + 8u * buf);
                ++acc_iter;
            }
        }
    }

    if constexpr (C_TMA) {
        // every TMA store of C must complete before the CTA exits
        if (warp >= 4 && lane == 0) bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

// ------------------------------------------------------------------ host ----

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Tensor map of a rows x k 16-bit operand with row pitch k_pitch elements,
// box = 64 elements (128 bytes) x box_rows, 128-byte swizzle; elements outside
// [0,k) x [0,rows) read as zero.
bool encode_operand_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t k, int64_t k_pitch,
                        int box_rows) {
    EncodeTiledFn enc = get_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(k_pitch) * 2u};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kTcBK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Opt in to the kernel's dynamic shared memory and ask for the largest
// shared-memory carveout, so that the CTAs per SM the planner counts on fit.
cudaError_t configure_kernel(const void* kern, size_t smem) {
    return kernel_attrs_once(kern, static_cast<int>(smem), true);
}

// Tensor map of C (m x n, 4-byte elements, row pitch ldc elements) for TMA
// stores: box 32 x 32, 128-byte swizzle.  Needs a 16-byte row pitch and base.
bool encode_c_map(CUtensorMap* map, void* ptr, int64_t m, int64_t n, int64_t ldc) {
    EncodeTiledFn enc = get_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(m)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldc) * 4u};
    cuuint32_t box[2] = {32u, 32u};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, ptr, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int BM, int BN, bool INT_OUT>
cudaError_t launch_one(const TcLaunch& a, cudaStream_t stream) {
    using Cfg = TcCfg<BM, BN>;
    CUtensorMap mA, mB;
    if (!encode_operand_map(&mA, a.A16, a.m, a.k, a.k_pitch, BM)) return cudaErrorInvalidValue;
    if (!encode_operand_map(&mB, a.B16, a.n, a.k, a.k_pitch, BN)) return cudaErrorInvalidValue;
    CUtensorMap mC;
    std::memset(&mC, 0, sizeof(mC));
    int c_tma = 0;
    const int64_t ldc = a.ldc > 0 ? a.ldc : a.n;
    if (ldc < a.n) return cudaErrorInvalidValue;
    // C may be absent only when every tile is requantised into rq.D
    const bool split = INT_OUT && a.split_k > 1;
    const bool requant = INT_OUT && a.rq.qmode != kQuantNone;
    if (a.C == nullptr && (!requant || split)) return cudaErrorInvalidValue;
    if (requant && (a.rq.D == nullptr || a.rq.row_scale == nullptr || a.rq.col_scale == nullptr))
        return cudaErrorInvalidValue;
    if (Cfg::TMA_STORE && a.C != nullptr && (ldc % 4) == 0 && (reinterpret_cast<uintptr_t>(a.C) % 16) == 0) {
        if (!encode_c_map(&mC, a.C, a.m, a.n, ldc)) return cudaErrorInvalidValue;
        c_tma = 1;
    }
    TcParams p;
    p.C = a.C;
    p.err = a.err;
    p.c_tma = c_tma;
    p.m = a.m;
    p.n = a.n;
    p.ldc = ldc;
    p.num_kb = static_cast<int>((a.k + kTcBK - 1) / kTcBK);
    p.chunk_kb = a.chunk_kb;
    p.tiles_m = static_cast<int>((a.m + BM - 1) / BM);
    p.tiles_n = static_cast<int>((a.n + BN - 1) / BN);
    p.tiles = p.tiles_m * p.tiles_n;
    p.split_k = a.split_k > 1 ? a.split_k : 1;
    p.split_from = p.split_k > 1 ? static_cast<int>(a.split_from) : p.tiles;
    p.units = p.split_from + (p.tiles - p.split_from) * p.split_k;
    p.rq = requant ? a.rq : RqOut{};
    auto kern = c_tma ? gemm_tc_kernel<BM, BN, INT_OUT, Cfg::TMA_STORE> : gemm_tc_kernel<BM, BN, INT_OUT, false>;
    cudaError_t e = configure_kernel(reinterpret_cast<const void*>(kern), Cfg::SMEM);
    if (e != cudaSuccess) return e;
    // programmatic dependent launch: set-up overlaps the kernel before; every
    // global access waits for it (pdl_wait)
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(a.grid), 1, 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, mA, mB, mC, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <bool INT_OUT>
cudaError_t dispatch(const TcLaunch& a, cudaStream_t stream) {
#define GEMM_TC_CASE(BM_, BN_) \
    if (a.bm == BM_ && a.bn == BN_) return launch_one<BM_, BN_, INT_OUT>(a, stream);
    GEMM_TC_CASE(128, 256)
    GEMM_TC_CASE(128, 128)
    GEMM_TC_CASE(128, 64)
    GEMM_TC_CASE(128, 32)
    GEMM_TC_CASE(64, 256)
    GEMM_TC_CASE(64, 128)
    GEMM_TC_CASE(64, 64)
    GEMM_TC_CASE(64, 32)
#undef GEMM_TC_CASE
    return cudaErrorInvalidValue;
}

template <int BM, int BN, bool INT_OUT>
const void* kernel_ptr() {
    return reinterpret_cast<const void*>(gemm_tc_kernel<BM, BN, INT_OUT, TcCfg<BM, BN>::TMA_STORE>);
}

const void* find_kernel(int bm, int bn, bool int_out) {
#define GEMM_TC_PTR(bm_, bn_)                                                                   \
    if (bm == bm_ && bn == bn_)                                                                 \
        return int_out ? kernel_ptr<bm_, bn_, true>() : kernel_ptr<bm_, bn_, false>();
    GEMM_TC_PTR(128, 256)
    GEMM_TC_PTR(128, 128)
    GEMM_TC_PTR(128, 64)
    GEMM_TC_PTR(128, 32)
    GEMM_TC_PTR(64, 256)
    GEMM_TC_PTR(64, 128)
    GEMM_TC_PTR(64, 64)
    GEMM_TC_PTR(64, 32)
#undef GEMM_TC_PTR
    return nullptr;
}

}  // namespace

bool tensor_map_encoder_available() { return get_encoder() != nullptr; }

void* tensor_map_encoder() { return reinterpret_cast<void*>(get_encoder()); }

cudaError_t launch_tc(const TcLaunch& a, cudaStream_t stream) {
    return a.int_out ? dispatch<true>(a, stream) : dispatch<false>(a, stream);
}

int tc_occupancy(int bm, int bn, bool int_out) {
    const void* k = find_kernel(bm, bn, int_out);
    if (!k) return 0;
    const size_t smem = tc_smem_bytes(bm, bn);
    if (configure_kernel(k, smem) != cudaSuccess) return 0;
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k, kTcThreads, smem) != cudaSuccess) return 0;
    return blocks;
}

int tc_num_regs(int bm, int bn, bool int_out) {
    const void* k = find_kernel(bm, bn, int_out);
    cudaFuncAttributes attr;
    if (!k || cudaFuncGetAttributes(&attr, k) != cudaSuccess) return -1;
    return attr.numRegs;
}

}  // namespace gemm
