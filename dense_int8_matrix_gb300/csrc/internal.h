// Internal declarations shared by the library's translation units (not part
// of the public C ABI in include/dense_int8_matrix.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/dense_int8_matrix.h"

namespace gemm {

// ---- the tensor-core kernel family (gemm_tc.cu) ---------------------------
// One CTA = 12 warps: warp 0 issues TMA copies, warp 1 owns TMEM and issues
// tcgen05.mma, warps 2-3 idle, warps 4-11 drain the accumulator (epilogue).
constexpr int kTcThreads = 384;
constexpr int kTcStages = 4;         // operand ring depth
constexpr int kTcBK = 64;            // K elements of a 16-bit operand per stage
constexpr int kTcRowBytes = 128;     // kTcBK * 2: one 128-byte swizzle row
constexpr int kTcEpilogueWarps = 8;

// int8 problems run on f16 tensor-core MMAs with fp32 accumulation.  Every
// int8 value and every product (|a*b| <= 2^14) is exact in f16 / fp32, and a
// fp32 sum of integers is exact while its magnitude stays within 2^24, i.e.
// for at most 2^24 / 2^14 = 1024 products.  So the accumulator is drained to
// int32 registers (exact) after every kI8ChunkK elements of K.
constexpr int kI8ChunkK = 1024;

constexpr int tc_tmem_cols(int bn) {
    int need = 2 * bn < 32 ? 32 : 2 * bn;
    int cols = 32;
    while (cols < need) cols *= 2;
    return cols;
}

// Wide tiles (BM = 128, BN >= 128) write C through shared memory and TMA
// stores: each epilogue warp stages 32 rows x 32 columns of 4-byte values
// (4 KiB, 128-byte swizzle) at a time.
constexpr bool tc_tma_store_tile(int bm, int bn) { return bm == 128 && bn >= 128; }
constexpr int kTcEpiStageBytes = 32 * 32 * 4;

constexpr size_t tc_smem_bytes(int bm, int bn) {
    // operand ring + epilogue staging + 1 KiB to align to the 1024-byte
    // swizzle atom + 1 KiB for barriers and flags
    return static_cast<size_t>(kTcStages) * (bm + bn) * kTcRowBytes +
           (tc_tma_store_tile(bm, bn) ? static_cast<size_t>(kTcEpilogueWarps) * kTcEpiStageBytes : 0) + 1024 + 1024;
}

// The two-SM tile (gemm_tc2.cu): a cluster of two CTAs computes 256 x 256 of
// C; per CTA a 6-stage ring of 128-row A and Bt halves (32 KiB per stage) and
// the same TMA-store epilogue staging as the wide one-SM tiles.
constexpr int kTc2Stages = 6;
constexpr size_t tc2_smem_bytes() {
    return static_cast<size_t>(kTc2Stages) * 2 * 128 * kTcRowBytes +
           static_cast<size_t>(kTcEpilogueWarps) * kTcEpiStageBytes + 1024 + 1024;
}

// Registers per thread the kernel is compiled for (launch bounds): wide
// tiles keep 64-128 running sums per epilogue thread and run one CTA per SM;
// narrow tiles fit two CTAs per SM.
constexpr int tc_regs_per_thread(int bn) { return bn >= 128 ? 168 : 80; }
constexpr int tc_min_blocks(int bn) { return bn >= 128 ? 1 : 2; }

// Tail split of the last, partial wave (int8 only).  With T tiles run by a
// persistent grid of G co-resident CTAs, R = T / G whole rounds run unsplit;
// the remaining T - R*G tiles are each split along K into S slices, S as large
// as fits the grid (S * tail <= G) and at most the number of K chunks (8 at
// most).  Returns S (1 = no split) and sets *split_from = R * G.
constexpr int kTcMaxSplit = 8;
inline int tc_tail_split(int64_t tiles, int64_t grid, int64_t nchunks, bool int_out, int64_t* split_from) {
    *split_from = tiles;
    if (!int_out || grid < 2 || tiles <= grid || nchunks < 2) return 1;
    const int64_t full = (tiles / grid) * grid;
    const int64_t tail = tiles - full;
    if (tail == 0) return 1;
    int64_t s = grid / tail;
    if (s > nchunks) s = nchunks;
    if (s > kTcMaxSplit) s = kTcMaxSplit;
    if (s < 2) return 1;
    *split_from = full;
    return static_cast<int>(s);
}

// The slices of a split tile all add their int32 partial sums into C (TMA
// reduce-add, or atomics), which the staging kernel has zeroed over those
// tiles: no slice waits on another, whatever order the CTAs run in.

// Order of the output tiles in both tensor kernels (and in the staging
// kernel's zeroing of split tiles): bands of kTcBandM M-tiles, N fastest
// inside a band, so CTAs running at the same time share A and Bt panels in L2.
constexpr int kTcBandM = 8;
__host__ __device__ inline void tc_tile_coords(int t, int tiles_m, int tiles_n, int& tm, int& tn) {
    const int per_band = kTcBandM * tiles_n;
    const int band = t / per_band;
    const int first_m = band * kTcBandM;
    const int rows_in_band = tiles_m - first_m < kTcBandM ? tiles_m - first_m : kTcBandM;
    const int local = t - band * per_band;
    tm = first_m + local % rows_in_band;
    tn = local / rows_in_band;
}

// Requantised output (gemm_i8_run_requant): D[i][j] = q((float(C[i][j]) *
// row_scale[i]) * col_scale[j]), q = bfloat16 or saturated int8 (requant.cuh).
enum { kQuantNone = 0, kQuantBf16 = 1, kQuantI8 = 2 };
struct RqOut {
    void* D = nullptr;                  // m x n bfloat16 (bit patterns) or int8
    const float* row_scale = nullptr;   // m floats, 16-byte aligned
    const float* col_scale = nullptr;   // n floats, 16-byte aligned
    int64_t ldd = 0;                    // row pitch of D in elements
    int qmode = kQuantNone;             // kQuant*
    int d_vec = 0;                      // 1: eight consecutive elements of a row take one 16-byte (bf16) / 8-byte (int8) store
};
// Tiles of a bm x bn tiling of C, [tile_from, tile_to) in tc_tile_coords
// order; bm == 0: all of C.
struct RqTiles {
    int bm = 0, bn = 0;
    int tiles_m = 0, tiles_n = 0;
    int tile_from = 0, tile_to = 0;
};
// The elementwise requant kernel (requant.cu): D over the tiles `t` from the
// int32 C (row pitch ldc), launched with programmatic stream serialization.
cudaError_t launch_requant(const int32_t* C, int64_t ldc, const RqOut& o, int64_t m, int64_t n, const RqTiles& t,
                           int num_sms, cudaStream_t stream);

struct TcLaunch {
    const void* A16;      // m x k_pitch 16-bit operand (f16 for int8 problems, bf16 otherwise)
    const void* A8 = nullptr;   // two-SM kernel, int8 problems: int8 A (m x k, k % 16 == 0) widened on chip
                                // instead of A16
    const void* B16;      // n x k_pitch 16-bit operand
    void* C;              // m x n int32 (int8 problems) or fp32
    int* err;             // device error word
    int64_t m, n, k, k_pitch;
    int bm, bn;
    int grid;
    int chunk_kb;         // k-blocks accumulated in TMEM before a drain
    bool int_out;         // true: int8 problem (f16 operands, int32 output)
    int split_k;          // K slices of the tail tiles (1 = none); C must be zero over those tiles
    int64_t split_from;   // first split tile
    int64_t ldc = 0;      // row pitch of C in elements (0: n)
    // int8 problems: whole tiles requantised into rq.D in the epilogue (split
    // tiles still add their int32 partial sums into C, which may then be
    // scratch); rq.qmode == kQuantNone: C as usual
    RqOut rq;
};

cudaError_t launch_tc(const TcLaunch& a, cudaStream_t stream);
// Two-SM kernel (bm = bn = 256); max_pairs = co-resident clusters (0: unknown).
cudaError_t launch_tc2(const TcLaunch& a, int max_pairs, cudaStream_t stream);
int tc2_max_pairs();
// Pairs launch_tc2 runs for a planned grid of 2 * pairs CTAs (declared again
// below, beside the tail split that uses it).
int tc2_pairs_for(int grid, int max_pairs, int64_t tiles);
int tc2_num_regs(bool int_out);
// block_per_cu of a tile as the planner counts it (registers, shared memory,
// TMEM); the tail split is used only when the whole grid fits at once.
int tc_blocks_per_sm(int bm, int bn);
// Occupancy of one kernel instance (CTAs per SM) as the runtime reports it.
int tc_occupancy(int bm, int bn, bool int_out);
int tc_num_regs(int bm, int bn, bool int_out);

// ---- operand staging (stage.cu) --------------------------------------------
// Int32 words of C that the staging kernel zeroes before a GEMM adds into
// them: all of C (bm == 0; the skinny path), or the tiles [tile_from, tile_to)
// of a bm x bn tiling in tc_tile_coords order (the tail split).
struct StageZero {
    int32_t* C = nullptr;   // nullptr: nothing to zero
    int64_t m = 0, n = 0;
    int bm = 0, bn = 0;
    int tiles_m = 0, tiles_n = 0;
    int tile_from = 0, tile_to = 0;
};

// K split of a tensor-path launch (tile bm x bn, persistent grid; for the
// two-SM tile over the pairs launch_tc2 runs): returns S (1 = none) and sets
// *split_from; `z` gets the split tiles of C for the staging kernel to zero.
// plan_split > 1 (int8): the plan splits every tile into that many K slices
// (whole K steps); otherwise only the tail of a partial last round is split.
int tc2_pairs_for(int grid, int max_pairs, int64_t tiles);
inline int tc_launch_split(int32_t* C, int64_t m, int64_t n, int64_t k, int bm, int bn, int grid, int chunk_kb,
                           bool int_out, int tc2_pairs, int plan_split, int64_t* split_from, StageZero* z) {
    const int tiles_m = static_cast<int>((m + bm - 1) / bm);
    const int tiles_n = static_cast<int>((n + bn - 1) / bn);
    const int64_t tiles = static_cast<int64_t>(tiles_m) * tiles_n;
    const int64_t num_kb = (k + kTcBK - 1) / kTcBK;
    const int64_t nchunks = (num_kb + chunk_kb - 1) / chunk_kb;
    int split;
    if (int_out && plan_split > 1) {
        split = plan_split < num_kb ? plan_split : static_cast<int>(num_kb);
        if (split > kTcMaxSplit) split = kTcMaxSplit;
        *split_from = 0;
    } else {
        const int64_t workers = bm == 256 ? tc2_pairs_for(grid, tc2_pairs, tiles) : grid;
        split = tc_tail_split(tiles, workers, nchunks, int_out, split_from);
    }
    *z = StageZero{};
    if (split > 1) {
        z->C = C;
        z->m = m;
        z->n = n;
        z->bm = bm;
        z->bn = bn;
        z->tiles_m = tiles_m;
        z->tiles_n = tiles_n;
        z->tile_from = static_cast<int>(*split_from);
        z->tile_to = static_cast<int>(tiles);
    } else {
        *split_from = tiles;
    }
    return split;
}
// int8 -> f16 (exact), row pitch k -> k_pitch, for A (m rows) and Bt (n rows),
// and the zeroing in `z`.  `err`: device error word of the bulk-copy
// variant's bounded waits (nullptr: that variant is not used).
cudaError_t launch_stage_i8(const int8_t* A, const int8_t* Bt, uint16_t* Ah, uint16_t* Bh, int64_t m,
                            int64_t n, int64_t k, int64_t k_pitch, const StageZero& z, int* err,
                            int num_sms, cudaStream_t stream);
// 16-bit copy with row pitch k -> k_pitch (bf16 problems whose k is not a
// multiple of 8).
cudaError_t launch_stage_b16(const uint16_t* A, const uint16_t* Bt, uint16_t* Ah, uint16_t* Bh, int64_t m,
                             int64_t n, int64_t k, int64_t k_pitch, int num_sms, cudaStream_t stream);

// ---- skinny path on the tensor cores (gemm_skinny_tc.cu) --------------------
// Needs k % 16 == 0 (TMA row pitch of int8 Bt) and 16-byte aligned A and Bt.
bool skinny_tc_supported(int64_t m, int64_t n, int64_t k, const void* A, const void* Bt);
// Its prologue (stage.cu): A (m x k int8, k % 16 == 0, A and A16 16-byte
// aligned) to f16 in A16 and all of C (m x n) zeroed, by one small CTA per SM
// that fits beside a running skinny CTA.  Launched with programmatic stream
// serialization, it becomes resident while the kernel before it still runs
// (and lets the skinny kernel after it launch), and touches memory only once
// that kernel has completed.
cudaError_t launch_skinny_prologue(const int8_t* A, uint16_t* A16, int32_t* C, int64_t m, int64_t n, int64_t k,
                                   int num_sms, cudaStream_t stream);
// A16: the m x k activations as f16 (row pitch k); C must be zero (the kernel
// adds its partial sums into it).
cudaError_t launch_skinny_tc(const int8_t* Bt, const uint16_t* A16, int32_t* C, int* err, int64_t m, int64_t n,
                             int64_t k, int num_sms, cudaStream_t stream);

// ---- skinny path on CUDA cores (gemm_skinny.cu) -----------------------------
cudaError_t launch_skinny_i8(const int8_t* A, const int8_t* Bt, int32_t* C, int64_t m, int64_t n, int64_t k,
                             int num_sms, cudaStream_t stream);

// ---- device error word and failure-detection self-test (selftest.cu) --------
// Device address of the current device's error word (a static __device__ int
// that every entry point's kernels write on a time-out and gemm_device_error
// reads); call with the device current and cache per device.
cudaError_t device_error_word(int** out);
// One CTA waits on an mbarrier that nothing completes; the bounded wait gives
// up after timeout_ns and records kDevErrTimeoutSelfTest in *err.
cudaError_t launch_selftest_wait(int* err, uint64_t timeout_ns, cudaStream_t stream);

// ---- driver entry point for tensor-map encoding (gemm_tc.cu) ----------------
bool tensor_map_encoder_available();
void* tensor_map_encoder();   // cuTensorMapEncodeTiled, or nullptr

// ---- argument checks shared by the entry points (api.cpp) -------------------
// A plan from gemm_*_plan (or edited to another compiled tile / grid) for
// `dtype`; GEMM_ERR_INVALID_ARG otherwise.
gemm_status check_plan(const gemm_plan* plan, int32_t dtype);
// Non-null device pointers, A and Bt 16-byte aligned, C 4-byte aligned.
gemm_status check_ptrs(const void* A, const void* Bt, const void* C);

// ---- kernel attributes (api.cpp) ---------------------------------------------
// Opts `kern` in to `smem_bytes` of dynamic shared memory (and, if asked, the
// largest shared-memory carveout) on the current device, once per device and
// kernel for the life of the process: cudaFuncSetAttribute costs host time on
// every call, which on short launches is more than the GPU time.
cudaError_t kernel_attrs_once(const void* kern, int smem_bytes, bool max_carveout);

}  // namespace gemm
