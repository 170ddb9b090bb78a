// Two-SM tensor-core GEMM (tcgen05 cta_group::2) for large problems.
//
// A cluster of two CTAs on two SMs computes one 256 x 256 tile of C.  Each
// CTA loads its own halves with TMA: 128 rows of A and 128 rows of Bt per
// 64-element K step (no multicast); one tcgen05.mma.cta_group::2 (M = 256,
// N = 256, K = 16), issued by the even CTA, reads the A rows of both CTAs
// and the B rows of both CTAs and leaves each CTA's 128 rows of the result
// in its own TMEM.  Per SM and K step that is 32 KB of operands through L2
// and shared memory instead of 48 KB for a one-SM 128 x 256 tile with the
// same output per SM, so the tensor pipe is fed more easily.  The TPU's
// 256 x 256 multiply-accumulate array ("文章导读: Motivation for and Evaluation
// of the First Tensor Processing Unit", section TPU介绍) has the same output
// block size.
//
// Roles (both CTAs, 12 warps each):
//   warp 0      TMA producer for this CTA's halves; the stage's "full"
//               barrier lives in the even CTA, whose producer also announces
//               the bytes of both CTAs;
//   warp 1      TMEM allocation (cta_group::2, both CTAs); in the even CTA
//               one lane issues the MMAs and commits with a multicast to
//               both CTAs' barriers (stage free, accumulator full);
//   warps 4-11  epilogue on this CTA's 128 rows, exactly as in the one-SM
//               kernel (int8: drain each 1024-element K chunk to exact int32;
//               TMA-store or vector-store C); releases the accumulator on the
//               even CTA's barrier.
//
// Widened A (int8 problems with k % 16 == 0, chosen by the caller for narrow
// C, where a staged f16 copy of A would cost more traffic than the multiply):
// int8 A is loaded by TMA (128 rows x 128 bytes, two K steps, per box) into a
// separate ring, and warps 2 and 3 of each CTA (one K step of each box) widen
// it exactly to f16 in the 128-byte swizzled layout of the operand ring, so A
// crosses HBM once, as int8; Bt still comes from the staged f16 copy.  The
// widened halves of both CTAs are announced on the even CTA's "full" barrier
// beside the TMA bytes of Bt.
//
// Tail split (int8 problems): when the last round of pairs is only partly
// filled, the tiles of that round run as split_k K slices on otherwise idle
// pairs.  The staging kernel zeroes C over those tiles, and every slice adds
// its exact int32 partial sums into C with a TMA reduce-add: no slice waits
// on another, whatever order the pairs run in.  When C's rows are not 16-byte
// aligned (no TMA), a pair's last unit uses its idle operand ring as staging
// for bulk copies or reduce-adds (a contiguous run of whole rows for odd
// n <= 256, row by row otherwise); earlier units go through the transposed
// 32 x 32 staging buffer into warp-wide atomics or stores.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "requant.cuh"

namespace gemm {

namespace {

constexpr int kT2Stages = kTc2Stages;
constexpr int kT2Half = 128;                      // rows of A and of Bt per CTA and K step
constexpr int kT2HalfBytes = kT2Half * kTcRowBytes;
constexpr int kT2StageBytes = 2 * kT2HalfBytes;   // this CTA's A and B halves
constexpr int kT2Cols = 256;                      // N of the pair tile = TMEM columns per accumulator
constexpr int kT2Half2 = kT2Cols / 2;             // columns per epilogue warp
constexpr int kT2EpiBytes = kTcEpilogueWarps * kTcEpiStageBytes;
constexpr size_t kT2Smem = static_cast<size_t>(kT2Stages) * kT2StageBytes + kT2EpiBytes + 1024 + 1024;
static_assert(kT2Smem == tc2_smem_bytes(), "shared-memory size known to the planner");

// Widened-A variant: a 4-stage f16 operand ring (filled by TMA for Bt and by
// the widening warps for A, on chip, so it needs little depth) and a 4-stage
// ring of int8 A (128 rows x 128 bytes = two K steps, 16 KiB, per stage and
// CTA) that covers the latency of the int8 stream from HBM.  Rows of 128
// bytes, not 64 (one K step), measured 8-12 % faster on GB300 at n <= 512
// (the TMA stream of 64-byte row pieces is the slower one).
constexpr int kT2WStages = 4;
constexpr int kT2W8Stages = 4;
constexpr int kT2W8Steps = 2;                      // K steps per int8 stage
constexpr int kT2W8Bytes = kT2Half * kT2W8Steps * kTcBK;   // 16 KiB
constexpr size_t kT2WSmem = static_cast<size_t>(kT2WStages) * kT2StageBytes +
                            static_cast<size_t>(kT2W8Stages) * kT2W8Bytes + kT2EpiBytes + 1024 + 1024;
static_assert(kT2WSmem <= 232448, "widened-A shared memory");

// Shared-memory rings of one kernel instance.  DEEP (widened A only): an
// instance for launches whose epilogue never stages C, i.e. whose every unit
// is its pair's last and goes out as a contiguous run (odd n <= 256, C's
// pitch n, no more units than pairs; the launch checks this): the 32 KiB of C
// staging go to a fifth f16 stage (measured on GB300: (4097, 16384, 255)
// 39.1 -> 37.5 us, (16384, 16384, 255) 102.2 -> 97.1 us).
template <bool WIDEN_A, bool DEEP = false>
struct T2Ring {
    static_assert(!DEEP || WIDEN_A, "the deep rings are a widened-A layout");
    static constexpr int STAGES = DEEP ? 5 : (WIDEN_A ? kT2WStages : kT2Stages);
    static constexpr int W8 = DEEP ? 3 : kT2W8Stages;   // int8 boxes
    static constexpr int EPI = DEEP ? 0 : kT2EpiBytes;  // C staging bytes
    static constexpr size_t SMEM = static_cast<size_t>(STAGES) * kT2StageBytes +
                                   (WIDEN_A ? static_cast<size_t>(W8) * kT2W8Bytes : 0) + EPI + 1024 + 1024;
};
static_assert(T2Ring<false>::SMEM == kT2Smem && T2Ring<true>::SMEM == kT2WSmem, "ring layouts");
static_assert(T2Ring<true, true>::SMEM <= 232448, "deep widened-A shared memory");

struct T2Params {
    void* C;
    int* err;
    int64_t m, n;
    int64_t ldc;                   // row pitch of C in elements
    int num_kb;
    int chunk_kb;
    int tiles_m, tiles_n, tiles;   // 256 x 256 tiles
    int units;                     // split_from + (tiles - split_from) * split_k
    int split_from;                // tiles [split_from, tiles) run as split_k K slices (C zeroed over them)
    int split_k;
    RqOut rq;                      // qmode != none: whole tiles requantised into rq.D, not written to C
};

// A unit of work: one tile over the K steps [kb_lo, kb_hi).  Units below
// split_from are whole tiles; above it, the slices of a split tile are
// consecutive units, each a run of whole K steps.
struct Unit2 {
    int tm, tn, kb_lo, kb_hi;
    int split_tile;   // index among the split tiles, -1 if the tile is whole
    int slice;
};

__device__ __forceinline__ Unit2 unit_at2(int u, const T2Params& p) {
    Unit2 x;
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

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// shared::cluster address of the same shared location in CTA `rank`
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// TMA load into this CTA's shared memory, completing on an mbarrier that may
// live in the peer CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* desc, int32_t x, int32_t y,
                                                 uint32_t bar_cluster, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(desc)), "r"(x), "r"(y), "r"(bar_cluster), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void mma_f16_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` (same offset) in both CTAs of the pair when the MMAs
// issued so far have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(mask)
        : "memory");
}

// Arrive on a barrier given by its shared::cluster address with the default
// (CTA-scope) release: the widening group's hand-off to the even CTA's MMA
// issuer, which then waits with the default acquire.  The widened bytes sit
// in the arriving CTA's own shared memory and are read there by its SM's half
// of the pair MMA; fence.proxy.async before the arrival orders them for the
// tensor core.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// Arrive on a barrier given by its shared::cluster address (possibly remote).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Write one 32-column slice of this warp's 32 rows of C, or add it into C
// (`add`, the slices of a split tile): each lane holds the 32 values of its
// row.  With C_TMA, the lanes fill the warp's 128B-swizzled 4 KiB staging
// buffer and one TMA store (or reduce-add) moves the 32 x 32 box (clipped at
// the edges of C); otherwise, with 16-byte-aligned rows, each lane stores
// its row, and with unaligned rows or adds the block is transposed through
// the staging buffer into coalesced stores or atomics along the rows.
template <bool C_TMA>
__device__ __forceinline__ void store_slice32(const CUtensorMap* tmC, const T2Params& p, const uint32_t (&r)[32],
                                              uint32_t stg, int lane, int row, int ytop, int cs, bool c_vec,
                                              bool add) {
    if constexpr (C_TMA) {
        const uint32_t row_base = stg + lane * 128;
        if (lane == 0) bulk_wait_read_all();   // the previous box has left the buffer
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c)
            st_shared_v4(row_base + ((c ^ (lane & 7)) << 4), r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (add)
                tma_reduce_add_2d(tmC, stg, cs, ytop);
            else
                tma_store_2d(tmC, stg, cs, ytop);
            bulk_commit();
        }
    } else if (c_vec && !add) {
        // 16-byte rows: each lane stores its row's 128 bytes
        if (row < p.m && cs + 32 <= p.n) {
            uint32_t* out = static_cast<uint32_t*>(p.C) + static_cast<int64_t>(row) * p.ldc + cs;
#pragma unroll
            for (int j = 0; j < 32; j += 4) *reinterpret_cast<uint4*>(out + j) = make_uint4(r[j], r[j + 1], r[j + 2], r[j + 3]);
        } else if (row < p.m) {
            uint32_t* out = static_cast<uint32_t*>(p.C) + static_cast<int64_t>(row) * p.ldc + cs;
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (cs + j < p.n) out[j] = r[j];
        }
    } else {
        // unaligned rows, or adds: the 32 x 32 block goes through the warp's
        // staging buffer so that every store (or atomic add) instruction
        // covers 32 consecutive columns of one row
        __syncwarp();   // the previous block has been read out
        stage_rows32(stg, lane, r);
        __syncwarp();
        const int col = cs + lane;
#pragma unroll 4
        for (int j = 0; j < 32; ++j) {
            const uint32_t v = staged_at(stg, j, lane);
            const int rr = ytop + j;
            if (rr < p.m && col < p.n) {
                uint32_t* o = static_cast<uint32_t*>(p.C) + static_cast<int64_t>(rr) * p.ldc + col;
                if (add)
                    atomicAdd(o, v);
                else
                    *o = v;
            }
        }
    }
}

// Row buffers for adding a split tile's last sums into C whose rows are not
// 16-byte aligned (no TMA): 128 values per row at a shift of 0-3 slots, in
// rows of 132 slots (528 bytes: the quarter-warp's eight 16-byte stores land
// in eight different bank groups), 32 rows per epilogue warp.  They reuse
// the operand rings (with the int8 ring behind the f16 one when A is widened
// on chip), which are idle once the CTA pair's last unit has left them.
constexpr int kT2RowSlots = kT2Half2 + 4;
constexpr int kT2RowBytes = kT2RowSlots * 4;
constexpr int kT2RowBufBytes = 32 * kT2RowBytes;
static_assert(kTcEpilogueWarps * kT2RowBufBytes <= kT2WStages * kT2StageBytes + kT2W8Stages * kT2W8Bytes &&
                  kTcEpilogueWarps * kT2RowBufBytes <= kT2Stages * kT2StageBytes,
              "row buffers fit in the operand rings");

// This lane's row of 128 sums into its row buffer, value c at slot c + A.
template <int A>
__device__ __forceinline__ void put_row_shifted(uint32_t buf, const int32_t (&acc)[kT2Half2]) {
#pragma unroll
    for (int i = 0; i < kT2RowSlots / 4; ++i) {
        uint32_t v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = 4 * i + j - A;
            v[j] = (c >= 0 && c < kT2Half2) ? static_cast<uint32_t>(acc[c]) : 0u;
        }
        st_shared_v4(buf + 16 * i, v[0], v[1], v[2], v[3]);
    }
}

// Add this lane's row of a split tile (128 columns from col0) into C: the
// 16-byte-aligned middle with one bulk reduce-add from the row buffer, the
// (at most three) values before and after it with atomics.  Columns past n
// and rows past m are not touched.
__device__ __forceinline__ void add_row_bulk(const T2Params& p, const int32_t (&acc)[kT2Half2], uint32_t buf, int row,
                                             int col0) {
    if (row >= p.m || col0 >= p.n) return;
    const int nv = static_cast<int>(min(static_cast<int64_t>(kT2Half2), p.n - col0));
    uint32_t* out = static_cast<uint32_t*>(p.C) + static_cast<int64_t>(row) * p.ldc + col0;
    const int a = static_cast<int>((reinterpret_cast<uintptr_t>(out) >> 2) & 3u);   // slots before out's 16-byte group
    switch (a) {
        case 0: put_row_shifted<0>(buf, acc); break;
        case 1: put_row_shifted<1>(buf, acc); break;
        case 2: put_row_shifted<2>(buf, acc); break;
        default: put_row_shifted<3>(buf, acc); break;
    }
    fence_proxy_async_smem();   // the bulk copy (async proxy) reads what this thread wrote
    const int lo = (a + 3) & ~3, hi = (a + nv) & ~3;   // aligned slots [lo, hi)
    if (hi > lo) {
        bulk_reduce_add_u32(out + (lo - a), buf + 4 * lo, static_cast<uint32_t>(4 * (hi - lo)));
        bulk_commit();
    }
    // the ends: slots [a, lo) and [max(hi, lo), a + nv)
    for (int t = a; t < lo && t < a + nv; ++t) atomicAdd(out + (t - a), ld_shared_u32(buf + 4 * t));
    for (int t = max(hi, lo); t < a + nv; ++t) atomicAdd(out + (t - a), ld_shared_u32(buf + 4 * t));
}

// Whole rows of C per tile (n <= 256, C's row pitch n): the 128 rows of a
// CTA's half tile are one contiguous run of C.  Each epilogue thread puts its
// row's sums into an image of that run in the idle operand ring (value j of
// the run at slot j + a, a = the run's start modulo 16 bytes, in elements),
// and once all eight epilogue warps have done so one thread moves the
// 16-byte-aligned middle with a few bulk copies, or bulk reduce-adds for a
// split tile, and the at most three values at each end with plain stores or
// atomics.  Rows past m are not in the run.
constexpr int kT2FlatPieces = 8;   // bulk operations per run
static_assert(kT2Half * kT2Cols * 4 + 16 <= kT2WStages * kT2StageBytes + kT2W8Stages * kT2W8Bytes &&
                  kT2Half * kT2Cols * 4 + 16 <= kT2Stages * kT2StageBytes &&
                  kT2Half * kT2Cols * 4 + 16 <=
                      T2Ring<true, true>::STAGES * kT2StageBytes + T2Ring<true, true>::W8 * kT2W8Bytes,
              "run image fits in the operand rings");

__device__ __forceinline__ int flat_shift(const T2Params& p, int row0) {
    const uint32_t* run = static_cast<const uint32_t*>(p.C) + static_cast<int64_t>(row0) * p.n;
    return static_cast<int>((reinterpret_cast<uintptr_t>(run) >> 2) & 3u);
}

__device__ __forceinline__ void put_flat(const T2Params& p, const int32_t (&acc)[kT2Half2], uint32_t img, int a,
                                         int row0, int row, int col0) {
    if (row >= p.m) return;
    const int nv = static_cast<int>(p.n) - col0;   // valid columns of this thread's 128
    const uint32_t base = img + 4u * static_cast<uint32_t>(a + (row - row0) * static_cast<int>(p.n) + col0);
#pragma unroll
    for (int c = 0; c < kT2Half2; ++c)
        if (c < nv) st_shared_u32(base + 4u * c, static_cast<uint32_t>(acc[c]));
}

__device__ __forceinline__ void move_flat(const T2Params& p, uint32_t img, int a, int row0, bool add) {
    const int rows = static_cast<int>(min(static_cast<int64_t>(kT2Half), p.m - row0));
    if (rows <= 0) return;
    const int count = rows * static_cast<int>(p.n);   // values in the run
    uint32_t* run = static_cast<uint32_t*>(p.C) + static_cast<int64_t>(row0) * p.n;
    const int lo = (a + 3) & ~3, hi = (a + count) & ~3;   // aligned slots [lo, hi)
    if (hi > lo) {
        const int per = 4 * ((hi - lo + 4 * kT2FlatPieces - 1) / (4 * kT2FlatPieces));   // >= 4 slots
        for (int s0 = lo; s0 < hi; s0 += per) {
            const int s1 = min(hi, s0 + per);
            if (add)
                bulk_reduce_add_u32(run + (s0 - a), img + 4u * s0, static_cast<uint32_t>(4 * (s1 - s0)));
            else
                bulk_store(run + (s0 - a), img + 4u * s0, static_cast<uint32_t>(4 * (s1 - s0)));
        }
        bulk_commit();
    }
    for (int t = a; t < a + count && t < lo; ++t) {
        const uint32_t v = ld_shared_u32(img + 4u * t);
        if (add) atomicAdd(run + (t - a), v); else run[t - a] = v;
    }
    for (int t = max(hi, lo); t < a + count; ++t) {
        const uint32_t v = ld_shared_u32(img + 4u * t);
        if (add) atomicAdd(run + (t - a), v); else run[t - a] = v;
    }
}

template <bool INT_OUT, bool C_TMA, bool WIDEN_A, bool DEEP>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const T2Params p) {
    static_assert(!WIDEN_A || INT_OUT, "A is widened from int8 only");
    static_assert(!DEEP || !C_TMA, "the deep rings have no C staging");
    using Ring = T2Ring<WIDEN_A, DEEP>;
    constexpr int kStages = Ring::STAGES;
    constexpr int kW8 = Ring::W8;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sA = base;
    const uint32_t sB = base + kStages * kT2HalfBytes;
    const uint32_t sA8 = base + kStages * kT2StageBytes;   // int8 A ring (widened-A variant)
    const uint32_t sEpi = sA8 + (WIDEN_A ? kW8 * kT2W8Bytes : 0);   // (DEEP: no C staging)
    uint8_t* ctrl = smem_raw + (sEpi - raw) + Ring::EPI;
    const uint32_t bar0 = smem_u32(ctrl);
    const uint32_t full_bar0 = bar0;                        // used in the even CTA
    const uint32_t empty_bar0 = bar0 + 8u * kStages;
    const uint32_t accf_bar0 = bar0 + 16u * kStages;
    const uint32_t acce_bar0 = accf_bar0 + 16u;             // used in the even CTA
    const uint32_t done_bar = acce_bar0 + 16u;
    const uint32_t a8full_bar0 = done_bar + 8u;             // [kW8] int8 A landed (local)
    const uint32_t a8empty_bar0 = a8full_bar0 + 8u * kW8;   // [kW8] int8 A read (local)
    const uint32_t flat_bar = a8empty_bar0 + 8u * kW8;      // the epilogue warps' run image is complete
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 8 * (2 * kStages + 5 + 2 * kW8 + 1));
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5;
    // the next kernel in the stream (the next call's staging kernel, which
    // waits for this one before it touches memory) may launch
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < kStages; ++s) {
            // widened A: the producer's arrival plus one per CTA's widening group
            mbar_init(full_bar0 + 8u * s, WIDEN_A ? 3 : 1);
            mbar_init(empty_bar0 + 8u * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar0 + 8u * b, 1);
            mbar_init(acce_bar0 + 8u * b, 2 * kTcEpilogueWarps);
        }
        mbar_init(done_bar, 1);
        mbar_init(flat_bar, kTcEpilogueWarps);
        if constexpr (WIDEN_A) {
            for (int s = 0; s < kW8; ++s) {
                mbar_init(a8full_bar0 + 8u * s, 1);
                mbar_init(a8empty_bar0 + 8u * s, kT2W8Steps);   // both widening warps
            }
        }
        *abort_flag = 0u;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), 2 * kT2Cols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();   // barriers and TMEM of both CTAs are ready
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer --
        if (WIDEN_A && lane == 1) {
            // int8 A into its own ring, gated only by the widening warps'
            // releases (not by the f16 slots), so the HBM stream runs up to
            // kW8 boxes ahead.  A unit's box j holds its K steps
            // kb_lo + 2j and kb_lo + 2j + 1 (the second unused past kb_hi)
            pdl_wait();
            const uint64_t pol = policy_evict_first();
            uint32_t issued = 0;
            bool ok = true;
            for (int u = pair; ok && u < p.units; u += npairs) {
                const Unit2 w = unit_at2(u, p);
                const int ya = w.tm * 256 + static_cast<int>(rank) * kT2Half;
                for (int kb = w.kb_lo; kb < w.kb_hi; kb += kT2W8Steps) {
                    const uint32_t s8 = issued % kW8, ph8 = (issued / kW8) & 1u;
                    if (!wait_bounded(a8empty_bar0 + 8u * s8, ph8 ^ 1u, abort_flag, p.err, kDevErrTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(a8full_bar0 + 8u * s8, kT2W8Bytes);
                    tma_load_2d(sA8 + s8 * kT2W8Bytes, &tmA, kb * kTcBK, ya, a8full_bar0 + 8u * s8, pol);
                    ++issued;
                }
            }
            // Teardown: the copies still in flight must land before the CTA
            // exits (earlier ones were waited for by the widening group
            // before their slot was reused)
            for (uint32_t j = issued > static_cast<uint32_t>(kW8) ? issued - kW8 : 0u; j < issued; ++j)
                wait_bounded(a8full_bar0 + 8u * (j % kW8), (j / kW8) & 1u, nullptr, p.err,
                             kDevErrTimeoutTeardown);
        } else if (lane == 0) {
            pdl_wait();   // the operands may come from the staging kernel just before
            const uint64_t pol = policy_evict_normal();
            uint32_t issued = 0;
            bool ok = true;
            for (int u = pair; ok && u < p.units; u += npairs) {
                const Unit2 w = unit_at2(u, p);
                const int ya = w.tm * 256 + static_cast<int>(rank) * kT2Half;
                const int yb = w.tn * 256 + static_cast<int>(rank) * kT2Half;
                for (int kb = w.kb_lo; kb < w.kb_hi; ++kb) {
                    const uint32_t s = issued % kStages;
                    const uint32_t ph = (issued / kStages) & 1u;
                    if (!wait_bounded(empty_bar0 + 8u * s, ph ^ 1u, abort_flag, p.err, kDevErrTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = map_to_rank(full_bar0 + 8u * s, 0);
                    if constexpr (WIDEN_A) {
                        // A comes from the widening warps (lane 1 streams the
                        // int8 bytes); only the bytes of Bt complete on the
                        // even CTA's barrier
                        if (leader) mbar_arrive_expect_tx(full_bar0 + 8u * s, 2 * kT2HalfBytes);
                    } else {
                        // both CTAs' copies complete on the even CTA's barrier,
                        // which expects the bytes of both
                        if (leader) mbar_arrive_expect_tx(full_bar0 + 8u * s, 2 * kT2StageBytes);
                        tma_load_2d_pair(sA + s * kT2HalfBytes, &tmA, kb * kTcBK, ya, fb, pol);
                    }
                    tma_load_2d_pair(sB + s * kT2HalfBytes, &tmB, kb * kTcBK, yb, fb, pol);
                    ++issued;
                }
            }
        }
    } else if (WIDEN_A && (warp == 2 || warp == 3)) {
        // --------------------------------------------- widen int8 A to f16 --
        // Warp 2 + h widens K step h of every int8 box (64 of its 128 bytes
        // per row): 128 rows x 64 int8 (sixteen 16-byte chunks per lane) ->
        // 128 rows x 64 f16 in the 128-byte swizzled layout the MMA
        // descriptor reads (chunk c of row r at ((c ^ (r & 7)) << 4)); the
        // int8 box has the same swizzle.  Lane l takes rows (l & 7) + 8i,
        // chunk l >> 3, so that each quarter-warp covers eight rows and every
        // 16-byte load and store is free of bank conflicts.  A box whose
        // second step lies past the unit's end is still released by warp 3.
        // Both warps wait on every int8 barrier phase in order; an f16 slot is
        // reused only after the MMA that read it, which needs this warp's own
        // earlier step, so no wait can fall two phases behind.
        const uint32_t h = static_cast<uint32_t>(warp - 2);
        uint32_t done = 0, box = 0;   // K steps and int8 boxes of the previous units
        bool ok = true;
        const uint32_t fb = map_to_rank(full_bar0, 0);
        const int cq = lane >> 3;
        for (int u = pair; ok && u < p.units; u += npairs) {
            const Unit2 w = unit_at2(u, p);
            const int steps = w.kb_hi - w.kb_lo;
            for (int rel = static_cast<int>(h); rel < steps; rel += kT2W8Steps) {
                const uint32_t d = done + static_cast<uint32_t>(rel);   // this K step, counted over units
                const uint32_t bx = box + static_cast<uint32_t>(rel / kT2W8Steps);
                const uint32_t s = d % kStages, ph = (d / kStages) & 1u;
                const uint32_t s8 = bx % kW8, ph8 = (bx / kW8) & 1u;
                int got = 1;
                if (lane == 0)
                    got = (wait_bounded(a8full_bar0 + 8u * s8, ph8, abort_flag, p.err, kDevErrTimeoutProducer) &&
                           wait_bounded(empty_bar0 + 8u * s, ph ^ 1u, abort_flag, p.err, kDevErrTimeoutProducer))
                              ? 1
                              : 0;
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) {
                    ok = false;
                    break;
                }
                const uint32_t src = sA8 + s8 * kT2W8Bytes;
                const uint32_t dst = sA + s * kT2HalfBytes;
                // all sixteen loads first (the shared-memory accesses are
                // volatile asm, which the compiler keeps in program order),
                // then widen and store
                uint4 v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int r = (lane & 7) + 8 * i;
                    v[i] = ld_shared_v4(src + r * 128 + (((4 * static_cast<int>(h) + cq) ^ (r & 7)) << 4));
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int r = (lane & 7) + 8 * i;
                    uint32_t wv[8];
                    widen16(v[i], wv);
                    const uint32_t row = dst + r * 128;
                    st_shared_v4(row + (((2 * cq) ^ (r & 7)) << 4), wv[0], wv[1], wv[2], wv[3]);
                    st_shared_v4(row + (((2 * cq + 1) ^ (r & 7)) << 4), wv[4], wv[5], wv[6], wv[7]);
                }
                fence_proxy_async_smem();   // the MMA (async proxy) reads what was just written
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(a8empty_bar0 + 8u * s8);
                    mbar_arrive_remote(fb + 8u * s);
                }
            }
            if (ok && (steps % kT2W8Steps) != 0 && h == 1) {
                // the unit's last box has no second step: release it unread
                const uint32_t bx = box + static_cast<uint32_t>(steps / kT2W8Steps);
                const uint32_t s8 = bx % kW8, ph8 = (bx / kW8) & 1u;
                if (lane == 0) {
                    if (wait_bounded(a8full_bar0 + 8u * s8, ph8, abort_flag, p.err, kDevErrTimeoutProducer))
                        mbar_arrive(a8empty_bar0 + 8u * s8);
                    else
                        ok = false;
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            }
            done += static_cast<uint32_t>(steps);
            box += static_cast<uint32_t>((steps + kT2W8Steps - 1) / kT2W8Steps);
        }
    } else if (warp == 1) {
        // ------------------------------------------- MMA issuer (even CTA) --
        if (lane == 0 && leader) {
            constexpr uint32_t idesc = idesc_f16(INT_OUT ? 0u : 1u, 256, kT2Cols);
            uint32_t consumed = 0, acc_iter = 0;
            bool ok = true;
            for (int u = pair; ok && u < p.units; u += npairs) {
                const Unit2 w = unit_at2(u, p);
                for (int c0 = w.kb_lo; ok && c0 < w.kb_hi; c0 += p.chunk_kb) {
                    const uint32_t buf = acc_iter & 1u;
                    const uint32_t aph = (acc_iter >> 1) & 1u;
                    if (!wait_bounded(acce_bar0 + 8u * buf, aph ^ 1u, abort_flag, p.err, kDevErrTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * kT2Cols;
                    const int c1 = min(w.kb_hi, c0 + p.chunk_kb);
                    for (int kb = c0; kb < c1; ++kb) {
                        const uint32_t s = consumed % kStages;
                        const uint32_t ph = (consumed / kStages) & 1u;
                        if (!wait_bounded(full_bar0 + 8u * s, ph, abort_flag, p.err, kDevErrTimeoutMma)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t adesc = smem_desc_sw128_kmajor(sA + s * kT2HalfBytes);
                        const uint64_t bdesc = smem_desc_sw128_kmajor(sB + s * kT2HalfBytes);
#pragma unroll
                        for (int kk = 0; kk < kTcBK / 16; ++kk)
                            mma_f16_ss_pair(d_tmem, adesc + 2u * kk, bdesc + 2u * kk, idesc,
                                            (kb > c0 || kk > 0) ? 1u : 0u);
                        mma_commit_pair(empty_bar0 + 8u * s);
                        ++consumed;
                    }
                    if (!ok) break;
                    mma_commit_pair(accf_bar0 + 8u * buf);
                    ++acc_iter;
                }
            }
            mma_commit_pair(done_bar);
            wait_bounded(done_bar, 0u, nullptr, p.err, kDevErrTimeoutTeardown);
        }
    } else if (warp >= 4) {
        // -------------------------------------------------------- epilogue --
        pdl_wait();   // C (zeroed over the split tiles by the staging kernel) only after the kernel before
        fence_proxy_async_global();   // TMA reduce-adds below follow that zeroing
        const int e = warp - 4;
        const int q = warp & 3;
        const int h = e >> 2;
        uint32_t acc_iter = 0;
        bool ok = true;
        const int row_in_tile = q * 32 + lane;
        const bool c_vec = ((p.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0);
        const uint32_t acce_leader = map_to_rank(acce_bar0, 0);
        const uint32_t stg = sEpi + e * kTcEpiStageBytes;
        for (int u = pair; ok && u < p.units; u += npairs) {
            const Unit2 w = unit_at2(u, p);
            // 32-bit coordinates, as in the TMA boxes (m, n < 2^31 - 256)
            const int row0 = w.tm * 256 + static_cast<int>(rank) * kT2Half;
            const int row = row0 + row_in_tile;
            const int col0 = w.tn * 256 + h * kT2Half2;
            const int ytop = row0 + q * 32;
            // int8 problems: exact int32 running sums over the K chunks
            int32_t acc[INT_OUT ? kT2Half2 : 1];
#pragma unroll
            for (int j = 0; j < (INT_OUT ? kT2Half2 : 1); ++j) acc[j] = 0;
            for (int c0 = w.kb_lo; c0 < w.kb_hi; c0 += p.chunk_kb) {
                const uint32_t buf = acc_iter & 1u;
                const uint32_t aph = (acc_iter >> 1) & 1u;
                const bool last = c0 + p.chunk_kb >= w.kb_hi;
                int got = 1;
                if (lane == 0)
                    got = wait_bounded(accf_bar0 + 8u * buf, aph, abort_flag, p.err, kDevErrTimeoutEpilogue) ? 1 : 0;
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tcol = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * kT2Cols + h * kT2Half2;
                if constexpr (INT_OUT) {
                    // drain the chunk into the running sums, then free the
                    // accumulator before any output work
#pragma unroll
                    for (int sl = 0; sl < kT2Half2 / 16; ++sl) {
                        uint32_t v[16];
                        tmem_ld_32x32b_x16(tcol + sl * 16, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            acc[sl * 16 + j] += __float2int_rn(__uint_as_float(v[j]));   // exact
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(acce_leader + 8u * buf);
                    ++acc_iter;
                    if (!last) continue;
                    if (p.rq.qmode != kQuantNone && w.split_tile < 0) {
                        // a whole tile: its exact sums are final, requantise them
                        // straight into D (eight columns per store)
                        const float rs = row < p.m ? __ldg(p.rq.row_scale + row) : 0.f;
#pragma unroll
                        for (int g = 0; g < kT2Half2 / 8; ++g) {
                            int32_t t[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j) t[j] = acc[g * 8 + j];
                            requant_store8(p.rq, p.m, p.n, row, col0 + g * 8, rs, t);
                        }
                        continue;
                    }
                    if constexpr (DEEP) {
                        if (!(p.tiles_n == 1 && (p.n & 1) && p.ldc == p.n && u + npairs >= p.units)) {
                            // not reached (the launch picks these rings only
                            // when every unit leaves as a run): with no C
                            // staging there is no other way out, so the call
                            // ends with an error and C incomplete
                            if (lane == 0) {
                                atomicCAS(p.err, 0, kDevErrTimeoutEpilogue);
                                *abort_flag = 1u;
                            }
                            continue;
                        }
                    }
                    if (!C_TMA && p.tiles_n == 1 && (p.n & 1) && p.ldc == p.n && u + npairs >= p.units) {
                        // the pair's last unit, and its tile holds whole rows
                        // of C: the operand ring is idle (all MMAs done), so
                        // this CTA's 128 rows go out as one run (odd n only:
                        // the lanes' rows then start in different banks of
                        // the image; even n would make its stores conflict)
                        const int a = flat_shift(p, row0);
                        put_flat(p, acc, sA, a, row0, row, col0);
                        fence_proxy_async_smem();   // the bulk copies (async proxy) read the image
                        __syncwarp();
                        if (lane == 0) mbar_arrive(flat_bar);
                        if (warp == 4 && lane == 0) {
                            if (wait_bounded(flat_bar, 0u, abort_flag, p.err, kDevErrTimeoutEpilogue))
                                move_flat(p, sA, a, row0, w.split_tile >= 0);
                        }
                        continue;
                    }
                    if (!C_TMA && w.split_tile >= 0 && u + npairs >= p.units) {
                        // the pair's last unit: its operand ring is idle (all
                        // MMAs done), so the rows go out by bulk reduce-add
                        add_row_bulk(p, acc, sA + e * kT2RowBufBytes + lane * kT2RowBytes, row, col0);
                        continue;
                    }
#pragma unroll
                    for (int sl = 0; sl < kT2Half2 / 32; ++sl) {
                        uint32_t r[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = static_cast<uint32_t>(acc[sl * 32 + j]);
                        store_slice32<C_TMA>(&tmC, p, r, stg, lane, row, ytop, col0 + sl * 32, c_vec,
                                             w.split_tile >= 0);
                    }
                } else {
                    // fp32 results (one chunk): load and store 32 columns at a time
#pragma unroll
                    for (int sl = 0; sl < kT2Half2 / 32; ++sl) {
                        uint32_t r[32];
                        tmem_ld_32x32b_x32(tcol + sl * 32, r);
                        tmem_wait_ld();
                        if (last) store_slice32<C_TMA>(&tmC, p, r, stg, lane, row, ytop, col0 + sl * 32, c_vec, false);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(acce_leader + 8u * buf);
                    ++acc_iter;
                }
            }
        }
    }

    if constexpr (C_TMA) {
        if (warp >= 4 && lane == 0) bulk_wait_all();
    } else {
        if (warp >= 4) bulk_wait_all();   // the rows' bulk reduce-adds (none issued is fine)
    }
    tc_fence_before();
    cluster_sync();   // the peer may still read this CTA's shared memory or barriers until here
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, 2 * kT2Cols);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool encode(CUtensorMap* map, CUtensorMapDataType type, void* ptr, uint64_t inner, uint64_t rows, uint64_t pitch_bytes,
            uint32_t box_inner, uint32_t box_rows) {
    auto enc = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {pitch_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    return enc(map, type, 2, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool INT_OUT, bool C_TMA, bool WIDEN_A = false, bool DEEP = false>
const void* tc2_kernel_ptr() {
    return reinterpret_cast<const void*>(gemm_tc2_kernel<INT_OUT, C_TMA, WIDEN_A, DEEP>);
}

cudaError_t configure2(const void* kern, size_t smem = kT2Smem) {
    return kernel_attrs_once(kern, static_cast<int>(smem), true);
}

// int8 A, m x k row-major (k % 16 == 0): 128-byte x 128-row boxes (two K
// steps), 128-byte swizzle; rows and K beyond the matrix read as zero.
bool encode_a8(CUtensorMap* map, const void* ptr, uint64_t k, uint64_t m) {
    auto enc = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
    if (!enc) return false;
    cuuint64_t dims[2] = {k, m};
    cuuint64_t strides[1] = {k};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kT2W8Steps * kTcBK), static_cast<cuuint32_t>(kT2Half)};
    cuuint32_t estr[2] = {1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int tc2_pairs_for(int grid, int max_pairs, int64_t tiles) {
    int64_t pairs = grid / 2;
    if (max_pairs > 0 && pairs > max_pairs) pairs = max_pairs;
    if (pairs > tiles) pairs = tiles;
    if (pairs < 1) pairs = 1;
    return static_cast<int>(pairs);
}

int tc2_max_pairs() {
    const void* k = tc2_kernel_ptr<true, true>();
    if (configure2(k) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = kT2Smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, k, &cfg) != cudaSuccess) return 0;
    return clusters;
}

cudaError_t launch_tc2(const TcLaunch& a, int max_pairs, cudaStream_t stream) {
    CUtensorMap mA, mB, mC;
    std::memset(&mC, 0, sizeof(mC));
    const bool widen = a.A8 != nullptr;
    if (widen && (!a.int_out || (a.k % 16) != 0 || (reinterpret_cast<uintptr_t>(a.A8) % 16) != 0))
        return cudaErrorInvalidValue;
    if (widen ? !encode_a8(&mA, a.A8, a.k, a.m)
              : !encode(&mA, CU_TENSOR_MAP_DATA_TYPE_UINT16, const_cast<void*>(a.A16), a.k, a.m, a.k_pitch * 2,
                        kTcBK, kT2Half))
        return cudaErrorInvalidValue;
    if (!encode(&mB, CU_TENSOR_MAP_DATA_TYPE_UINT16, const_cast<void*>(a.B16), a.k, a.n, a.k_pitch * 2, kTcBK, kT2Half))
        return cudaErrorInvalidValue;
    const int64_t ldc = a.ldc > 0 ? a.ldc : a.n;
    if (ldc < a.n) return cudaErrorInvalidValue;
    // C may be absent only when every tile is requantised into rq.D
    const bool requant = a.int_out && a.rq.qmode != kQuantNone;
    if (a.C == nullptr && (!requant || (a.split_k > 1 && a.split_from < (a.m + 255) / 256 * ((a.n + 255) / 256))))
        return cudaErrorInvalidValue;
    if (requant && (a.rq.D == nullptr || a.rq.row_scale == nullptr || a.rq.col_scale == nullptr))
        return cudaErrorInvalidValue;
    // (no C at all: requantised output without split tiles)
    const bool c_tma = a.C != nullptr && (ldc % 4) == 0 && (reinterpret_cast<uintptr_t>(a.C) % 16) == 0;
    if (c_tma && !encode(&mC, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.C, a.n, a.m, ldc * 4, 32, 32))
        return cudaErrorInvalidValue;
    T2Params p;
    p.C = a.C;
    p.err = a.err;
    p.m = a.m;
    p.n = a.n;
    p.ldc = ldc;
    p.num_kb = static_cast<int>((a.k + kTcBK - 1) / kTcBK);
    p.chunk_kb = a.chunk_kb;
    p.tiles_m = static_cast<int>((a.m + 255) / 256);
    p.tiles_n = static_cast<int>((a.n + 255) / 256);
    p.tiles = p.tiles_m * p.tiles_n;
    // the split was planned for this number of pairs; units only reorder the
    // work, so any pair count stays correct
    const bool split = a.int_out && a.split_k > 1 && a.split_from < p.tiles;
    p.split_k = split ? a.split_k : 1;
    p.split_from = split ? static_cast<int>(a.split_from) : p.tiles;
    p.units = p.split_from + (p.tiles - p.split_from) * p.split_k;
    p.rq = requant ? a.rq : RqOut{};
    const int pairs = tc2_pairs_for(a.grid, max_pairs, p.units);
    // the deep widened-A rings: every unit is its pair's last (units <= pairs)
    // and leaves as a contiguous run of whole rows (odd n <= 256, pitch n)
    const bool deep = widen && !c_tma && p.tiles_n == 1 && (a.n & 1) && ldc == a.n && p.units <= pairs;
    const void* kern = deep ? tc2_kernel_ptr<true, false, true, true>()
                       : widen ? (c_tma ? tc2_kernel_ptr<true, true, true>() : tc2_kernel_ptr<true, false, true>())
                       : a.int_out ? (c_tma ? tc2_kernel_ptr<true, true>() : tc2_kernel_ptr<true, false>())
                                   : (c_tma ? tc2_kernel_ptr<false, true>() : tc2_kernel_ptr<false, false>());
    const size_t smem = deep ? T2Ring<true, true>::SMEM : widen ? kT2WSmem : kT2Smem;
    cudaError_t e = configure2(kern, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic dependent launch: set-up overlaps the kernel before; every
    // global access waits for it (pdl_wait)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    void* args[] = {&mA, &mB, &mC, &p};
    e = cudaLaunchKernelExC(&cfg, kern, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

int tc2_num_regs(bool int_out) {
    cudaFuncAttributes attr;
    const void* k = int_out ? tc2_kernel_ptr<true, true>() : tc2_kernel_ptr<false, true>();
    if (cudaFuncGetAttributes(&attr, k) != cudaSuccess) return -1;
    return attr.numRegs;
}

}  // namespace gemm
