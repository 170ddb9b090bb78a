// Skinny int8 GEMM on the tensor cores (m <= 128): C = A x B with B stored
// K-major as Bt (n x k).  Bt (n*k bytes) dwarfs A and C, so the kernel's job is
// to stream Bt from HBM once, at full bandwidth; the patent CN114238853A
// (claim 4 S3) calls such shapes too small to fill the chip with output tiles.
//
// Computed as C^T = Bt x A^T ("swap AB"): the MMA's M side is 128 rows of Bt,
// its N side is m padded to NP in {16, 32, 64, 128}, fp32 accumulation in TMEM,
// drained to exact int32 every 1024 K elements as in the large kernel.
//
// A pipeline stage is 256 K elements (four K steps of 64): every Bt row is
// fetched as 256 contiguous bytes (two 128-byte TMA boxes), which a stream of
// short row fragments cannot match (measured on GB300: 64-byte rows stream
// at ~4.3 TB/s, 128-byte rows at ~6.5 TB/s, 256-byte rows at ~6.9 TB/s).
//
// Roles, per CTA (20 warps):
//   warp 0      TMA: the int8 Bt boxes (128 rows x 256 B, 128-byte swizzle)
//               into a 3-deep ring;
//   warp 2      TMA: the f16 activation boxes (NP rows x 256 K) into a
//               2-6-deep ring (they are re-read by every CTA and stay in L2);
//   warps 4-11  two groups of four warps that take the stages in turn (one
//               warp of a group per TMEM lane quarter): each lane reads its
//               Bt row (256 int8) from shared memory, releases the stage,
//               widens the row to f16 in registers (exact) and writes it with
//               tcgen05.st into one of three 128-column TMEM operand buffers
//               (two for NP = 128, whose accumulators take 256 columns).
//               Shared memory carries only the int8 bytes, read once;
//   warps 1, 3  one thread each issues the tcgen05.mma of alternate stages
//               (A from TMEM, B = activations from shared memory): a small-N
//               MMA costs ~45 cycles of issue whatever N, so two issuers keep
//               the tensor pipe fed while each waits for its next stage;
//   warps 12-19 drain each accumulator chunk (two warps per lane quarter,
//               half of the NP columns each) into registers, zero and
//               release the accumulator, then convert the chunk to int32
//               (exact) and add it into C (pre-zeroed) with coalesced
//               integer atomics (exact and order-free).
// Work split ("stream-K"): the (128-row tile, stage) iterations are numbered
// tile-major and every CTA takes an equal contiguous range, so all SMs
// stream the same number of Bt bytes.
//
// Back-to-back calls overlap (programmatic dependent launch): every CTA lets
// the next kernel in the stream launch as soon as it starts, so the next
// call's prologue (A to f16, C zeroed: one small CTA per SM beside this one)
// is resident and waiting before this kernel ends.  The skinny kernel behind
// that prologue launches as this one ends (measured on GB300: only one
// kernel runs ahead of an unfinished one) and its CTAs take the SMs as they
// free; each sets up, and loads Bt and its activations and adds into C only
// after its grid dependency wait.
//
// Ring depths, measured on GB300 in back-to-back calls (k = n = 8192): a
// shallow Bt ring is faster.  A call is bound by the latency of its first
// stages, not by the stream (which runs at DRAM rate either way), and a deep
// ring makes every CTA queue its whole ring at once: m = 1 with 6 / 4 / 3 / 2
// stages 17.7 / 17.3 / 16.5 / 18.5 us per call, m = 64 with 5 / 3 stages
// (activation slots 2 / 4) 21.6 / 20.2 us.  Prefetching the first Bt stages
// into L2 before the wait cost time on top (m = 1, 3 stages: 17.1 us with 4
// stages ahead, 17.0 with 12, 16.5 with none).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace gemm {

namespace {

constexpr int kSkKbPerStage = 4;                     // K steps of 64 per stage
constexpr int kSkBtBox = 128 * 128;                  // one 128 B x 128-row box
constexpr int kSkBtStage = 2 * kSkBtBox;             // 256 B x 128 rows
constexpr int kSkGroups = 2;                         // widening groups (4 warps each)
// Barriers that two alternating warps (issuers or widening groups) would wait
// on at alternate phases are kept apart instead: a parity wait can only tell
// two neighbouring phases apart, so every barrier must have one waiter
// sequence.  Operand-buffer barriers are indexed by stage mod 2 x buffers
// (buffer x issuer), the Bt ring's "full" barriers by stage mod 2 x ring
// depth.
constexpr int kSkEpiWarps = 8;
constexpr int kSkWidenWarp0 = 4;
constexpr int kSkEpiWarp0 = kSkWidenWarp0 + 4 * kSkGroups;
constexpr int kSkThreads = 32 * (kSkEpiWarp0 + kSkEpiWarps);   // 640
constexpr int kSkChunkStages = kI8ChunkK / (64 * kSkKbPerStage);  // stages per exact fp32 chunk

template <int NP>
struct SkCfg {
    static constexpr int ACT_BOX = NP * 128;                   // f16 activation box: 64 K x NP rows
    static constexpr int ACT_STAGE = kSkKbPerStage * ACT_BOX;
    // TMEM: ABUFS operand buffers of 128 columns and two NP-column accumulators.
    static constexpr int ABUFS = NP >= 128 ? 2 : 3;
    static constexpr int ABUF_BARS = 2 * ABUFS;
    // Three Bt stages (see the measurements above); the activation ring gets
    // the room left, an even number of slots so that each slot always serves
    // the same MMA issuer (NP = 128 activation stages are 64 KB).
    static constexpr int BT_STAGES = 3;
    static constexpr int ACT_STAGES = NP >= 128 ? 2 : (NP == 32 ? 6 : 4);
    static constexpr int TMEM_COLS = 512;
    static constexpr int EPI_COLS = NP / 2;                    // columns per epilogue warp
    // barriers (8 B each), the TMEM address and the abort flag
    static constexpr int CTRL = 8 * (3 * BT_STAGES + 2 * ACT_STAGES + 2 * ABUF_BARS + 5) + 8;
    // + up to 1023 B to align the ring to the 1024 B the 128-byte swizzle needs
    static constexpr size_t SMEM =
        static_cast<size_t>(BT_STAGES) * kSkBtStage + static_cast<size_t>(ACT_STAGES) * ACT_STAGE + 512 + 1024;
    static_assert(ABUFS * 128 + 2 * NP <= TMEM_COLS, "TMEM budget");
    static_assert(CTRL <= 512, "control block");
    // with the 1 KiB the SM reserves per CTA, one skinny CTA and one prologue
    // CTA fit in the SM's 228 KiB of shared memory
    static_assert(SMEM + 1024 + 1024 <= 233472, "shared memory");
};

struct SkParams {
    int32_t* C;
    int* err;
    int m, n;
    int num_sb;       // stages of 256 K per tile
    int tiles;        // ceil(n / 128)
    int64_t iters;    // tiles * num_sb
    int iters32;      // iters * grid fits 32 bits
};

__device__ __forceinline__ void cta_range(const SkParams& p, int64_t& lo, int64_t& hi) {
    if (p.iters32) {   // iters * grid < 2^32: 32-bit arithmetic (cheaper at start-up)
        const uint32_t it = static_cast<uint32_t>(p.iters);
        lo = it * blockIdx.x / gridDim.x;
        hi = it * (blockIdx.x + 1) / gridDim.x;
    } else {
        lo = p.iters * blockIdx.x / gridDim.x;
        hi = p.iters * (blockIdx.x + 1) / gridDim.x;
    }
}

// Position of an iteration: its 128-row tile and its stage within the tile,
// advanced incrementally (no division inside the loops).
struct Cursor {
    int tile, sb;
    __device__ __forceinline__ void advance(int num_sb) {
        if (++sb == num_sb) {
            sb = 0;
            ++tile;
        }
    }
};

__device__ __forceinline__ Cursor cursor_at(const SkParams& p, int64_t i) {
    Cursor c;
    if (p.iters32) {
        const uint32_t u = static_cast<uint32_t>(i);
        c.tile = static_cast<int>(u / static_cast<uint32_t>(p.num_sb));
        c.sb = static_cast<int>(u - static_cast<uint32_t>(c.tile) * static_cast<uint32_t>(p.num_sb));
    } else {
        c.tile = static_cast<int>(i / p.num_sb);
        c.sb = static_cast<int>(i - static_cast<int64_t>(c.tile) * p.num_sb);
    }
    return c;
}

// A chunk ends after a stage that closes 1024 K elements of a tile, the
// tile, or the CTA's range (`last`).
__device__ __forceinline__ bool chunk_ends(const SkParams& p, const Cursor& c, bool last) {
    return last || (c.sb + 1 == p.num_sb) || ((c.sb + 1) % kSkChunkStages == 0);
}

template <int NP>
__global__ void __launch_bounds__(kSkThreads, 1)
    skinny_tc_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmA,
                     const SkParams p) {
    using Cfg = SkCfg<NP>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sBt = base;
    const uint32_t sAct = base + Cfg::BT_STAGES * kSkBtStage;
    uint8_t* ctrl = smem_raw + (base - raw) + Cfg::BT_STAGES * kSkBtStage + Cfg::ACT_STAGES * Cfg::ACT_STAGE;
    const uint32_t bar0 = smem_u32(ctrl);
    constexpr uint32_t kFullB = 2 * Cfg::BT_STAGES;           // "full" barriers of the Bt ring
    const uint32_t fullB0 = bar0;                              // [2 * BT_STAGES], stage n: n % (2 * BT_STAGES)
    const uint32_t emptyB0 = fullB0 + 8u * kFullB;             // [BT_STAGES], stage n: n % BT_STAGES
    const uint32_t fullA0 = emptyB0 + 8u * Cfg::BT_STAGES;     // [ACT_STAGES]
    const uint32_t emptyA0 = fullA0 + 8u * Cfg::ACT_STAGES;    // [ACT_STAGES]
    constexpr uint32_t kAbufs = Cfg::ABUFS, kAbufBars = Cfg::ABUF_BARS;
    const uint32_t aready0 = emptyA0 + 8u * Cfg::ACT_STAGES;   // [ABUF_BARS], stage n: n % ABUF_BARS
    const uint32_t afree0 = aready0 + 8u * kAbufBars;          // [ABUF_BARS], stage n: n % ABUF_BARS
    const uint32_t accf0 = afree0 + 8u * kAbufBars;            // [2]
    const uint32_t acce0 = accf0 + 16u;                        // [2]
    const uint32_t done_bar = acce0 + 16u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(
        ctrl + 8 * (kFullB + Cfg::BT_STAGES + 2 * Cfg::ACT_STAGES + 2 * kAbufBars + 5));
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // the next kernel in the stream (the next call's prologue) may launch
    pdl_launch_dependents();

    if (warp == 0 && lane == 0) {
        // the descriptors are fetched while the CTA sets up
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmA);
        for (uint32_t s = 0; s < kFullB; ++s) mbar_init(fullB0 + 8u * s, 1);
        for (int s = 0; s < Cfg::BT_STAGES; ++s) mbar_init(emptyB0 + 8u * s, 4);   // the widening group's warps
        for (int s = 0; s < Cfg::ACT_STAGES; ++s) {
            mbar_init(fullA0 + 8u * s, 1);
            mbar_init(emptyA0 + 8u * s, 1);   // the MMA's commit
        }
        for (uint32_t b = 0; b < kAbufBars; ++b) {
            mbar_init(aready0 + 8u * b, 4);
            mbar_init(afree0 + 8u * b, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8u * b, 2);   // one arrival per MMA issuer
            mbar_init(acce0 + 8u * b, kSkEpiWarps);
        }
        mbar_init(done_bar, 2);
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
    const uint32_t tmem_acc = tmem_base + kAbufs * 128;     // two accumulators of NP columns

    int64_t lo, hi;
    cta_range(p, lo, hi);

    if (warp == 0) {
        // ------------------------------------------------------- TMA: Bt --
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            pdl_wait();   // the kernel before may still be running (and writing Bt)
            uint32_t n_iss = 0;
            Cursor c = cursor_at(p, lo);
            for (int64_t i = lo; i < hi; ++i, ++n_iss, c.advance(p.num_sb)) {
                const uint32_t s = n_iss % Cfg::BT_STAGES, ph = (n_iss / Cfg::BT_STAGES) & 1u;
                if (!wait_bounded(emptyB0 + 8u * s, ph ^ 1u, abort_flag, p.err, kDevErrTimeoutProducer)) break;
                const int tile = c.tile;
                const int x = c.sb * 256;
                const uint32_t dst = sBt + s * kSkBtStage;
                const uint32_t fb = fullB0 + 8u * (n_iss % kFullB);
                mbar_arrive_expect_tx(fb, kSkBtStage);
                tma_load_2d(dst, &tmB, x, tile * 128, fb, pol);
                tma_load_2d(dst + kSkBtBox, &tmB, x + 128, tile * 128, fb, pol);
            }
            // the last BT_STAGES copies may still be in flight (earlier ones
            // landed before their slot was reused)
            for (uint32_t j = n_iss > static_cast<uint32_t>(Cfg::BT_STAGES) ? n_iss - Cfg::BT_STAGES : 0u; j < n_iss; ++j)
                wait_bounded(fullB0 + 8u * (j % kFullB), (j / kFullB) & 1u, nullptr, p.err, kDevErrTimeoutTeardown);
        }
    } else if (warp == 2) {
        // ---------------------------------------------- TMA: activations --
        if (lane == 0) {
            pdl_wait();   // the activations are written by the prologue just before
            const uint64_t pol = policy_evict_last();
            uint32_t n_iss = 0;
            Cursor c = cursor_at(p, lo);
            for (int64_t i = lo; i < hi; ++i, ++n_iss, c.advance(p.num_sb)) {
                const uint32_t s = n_iss % Cfg::ACT_STAGES, ph = (n_iss / Cfg::ACT_STAGES) & 1u;
                if (!wait_bounded(emptyA0 + 8u * s, ph ^ 1u, abort_flag, p.err, kDevErrTimeoutProducer)) break;
                const int kb0 = c.sb * kSkKbPerStage;
                const uint32_t dst = sAct + s * Cfg::ACT_STAGE;
                mbar_arrive_expect_tx(fullA0 + 8u * s, Cfg::ACT_STAGE);
#pragma unroll
                for (int j = 0; j < kSkKbPerStage; ++j)
                    tma_load_2d(dst + j * Cfg::ACT_BOX, &tmA, (kb0 + j) * 64, 0, fullA0 + 8u * s, pol);
            }
            for (uint32_t s = 0; s < static_cast<uint32_t>(Cfg::ACT_STAGES) && s < n_iss; ++s) {
                const uint32_t last = s + ((n_iss - 1u - s) / Cfg::ACT_STAGES) * Cfg::ACT_STAGES;
                wait_bounded(fullA0 + 8u * s, (last / Cfg::ACT_STAGES) & 1u, nullptr, p.err, kDevErrTimeoutTeardown);
            }
        }
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------------------------ MMA --
        // Two issuers take the stages in turn (warp 1: even, warp 3: odd) and
        // add into the chunk's pre-zeroed accumulator (integer sums are
        // order-free), so one issues while the other waits.  At every chunk
        // end each issuer arrives once on accf: by commit if it issued MMAs in
        // the chunk, by a plain arrival otherwise.
        if (lane == 0) {
            const uint32_t g = warp == 1 ? 0u : 1u;
            constexpr uint32_t idesc = idesc_f16(0u, 128, NP);
            bool ok = true;
            uint32_t ch = 0;
            bool issued_in_chunk = false, acc_ready = false;
            Cursor c = cursor_at(p, lo);
            uint32_t n = 0;
            for (int64_t i = lo; i < hi; ++i, ++n, c.advance(p.num_sb)) {
                const uint32_t buf = ch & 1u;
                if (ok && (n & 1u) == g) {
                    const uint32_t sa = n % Cfg::ACT_STAGES, pha = (n / Cfg::ACT_STAGES) & 1u;
                    const uint32_t b = n % kAbufs;
                    const uint32_t rb = n % kAbufBars, rph = (n / kAbufBars) & 1u;
                    ok = (acc_ready || wait_bounded(acce0 + 8u * buf, (ch >> 1) & 1u, abort_flag, p.err,
                                                    kDevErrTimeoutMma)) &&
                         wait_bounded(fullA0 + 8u * sa, pha, abort_flag, p.err, kDevErrTimeoutMma) &&
                         wait_bounded(aready0 + 8u * rb, rph, abort_flag, p.err, kDevErrTimeoutMma);
                    if (ok) {
                        acc_ready = true;
                        tc_fence_after();
                        const uint32_t d_tmem = tmem_acc + buf * NP;
                        const uint32_t a_tmem = tmem_base + b * 128;
                        const uint32_t act = sAct + sa * Cfg::ACT_STAGE;
#pragma unroll
                        for (int j = 0; j < kSkKbPerStage; ++j) {
                            const uint64_t bdesc = smem_desc_sw128_kmajor(act + j * Cfg::ACT_BOX);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_f16_ts(d_tmem, a_tmem + j * 32 + kk * 8, bdesc + 2u * kk, idesc, 1u);
                        }
                        mma_commit(afree0 + 8u * rb);
                        mma_commit(emptyA0 + 8u * sa);
                        issued_in_chunk = true;
                    }
                }
                if (chunk_ends(p, c, i + 1 == hi)) {
                    // An issuer with no stage in this chunk still arrives, but
                    // only once the epilogue has drained this accumulator's
                    // previous chunk: otherwise its (immediate) arrival could
                    // complete that earlier phase before the other issuer's
                    // MMAs into it have finished.
                    if (ok && !acc_ready)
                        ok = wait_bounded(acce0 + 8u * buf, (ch >> 1) & 1u, abort_flag, p.err, kDevErrTimeoutMma);
                    if (ok) {
                        if (issued_in_chunk)
                            mma_commit(accf0 + 8u * buf);
                        else
                            mbar_arrive(accf0 + 8u * buf);
                    }
                    issued_in_chunk = false;
                    acc_ready = false;
                    ++ch;
                }
            }
            // Teardown: every MMA issued must complete before TMEM is freed.
            mma_commit(done_bar);
            wait_bounded(done_bar, 0u, nullptr, p.err, kDevErrTimeoutTeardown);
        }
    } else if (warp >= kSkWidenWarp0 && warp < kSkEpiWarp0) {
        // ---------------------------------------------------------- widen --
        const int q = warp & 3;
        const int g = (warp - kSkWidenWarp0) >> 2;   // this warp's group: stages n = g mod kSkGroups
        const int row = q * 32 + lane;                // row of the 128-row Bt box
        const uint32_t swz = row & 7;                 // 128-byte swizzle of this row
        uint32_t n = g;
        for (int64_t i = lo + g; i < hi; i += kSkGroups, n += kSkGroups) {
            const uint32_t s = n % Cfg::BT_STAGES;
            const uint32_t b = n % kAbufs;
            int got = 1;
            if (lane == 0) {
                got = wait_bounded(fullB0 + 8u * (n % kFullB), (n / kFullB) & 1u, abort_flag, p.err,
                                   kDevErrTimeoutEpilogue);
                // buffer b last held stage n - ABUFS: its MMAs must be complete
                if (got && n >= kAbufs) {
                    const uint32_t pn = n - kAbufs;
                    got = wait_bounded(afree0 + 8u * (pn % kAbufBars), (pn / kAbufBars) & 1u, abort_flag, p.err,
                                       kDevErrTimeoutEpilogue);
                }
            }
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) break;
            tc_fence_after();
            // the row's 256 bytes: box 0 holds K 0..127, box 1 K 128..255
            uint4 v[16];
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) {
                const uint32_t src = sBt + s * kSkBtStage + (cc >> 3) * kSkBtBox + row * 128;
                v[cc] = ld_shared_v4(src + (((cc & 7) ^ swz) << 4));
            }
            // the bytes are in registers: the stage can be refilled
            __syncwarp();
            if (lane == 0) mbar_arrive(emptyB0 + 8u * s);
            const uint32_t dst = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + b * 128;
#pragma unroll
            for (int hf = 0; hf < 8; ++hf) {
                uint32_t w[16];
                widen16(v[2 * hf], w);
                widen16(v[2 * hf + 1], w + 8);
                tmem_st_32x32b_x16(dst + hf * 16, w);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(aready0 + 8u * (n % kAbufBars));
        }
    } else if (warp >= kSkEpiWarp0) {
        // ------------------------------------------------------- epilogue --
        // Every drained chunk (at most 1024 K elements, an exact integer in
        // fp32) is added into C at once, and the accumulator is zeroed for its
        // next chunk (the MMAs only ever accumulate).
        const int q = warp & 3;
        const int half = (warp - kSkEpiWarp0) >> 2;   // which half of the NP columns
        const int col0 = half * Cfg::EPI_COLS;
        const int jrow = q * 32 + lane;           // TMEM lane = row of the Bt tile = column j of C
        const int rows = min(Cfg::EPI_COLS, p.m - col0);
        const uint32_t lanes = static_cast<uint32_t>(q * 32) << 16;
        uint32_t zero[16];
#pragma unroll
        for (int z = 0; z < 16; ++z) zero[z] = 0u;
        // both accumulators start at zero
#pragma unroll
        for (int bz = 0; bz < 2; ++bz)
#pragma unroll
            for (int c0 = 0; c0 < Cfg::EPI_COLS; c0 += 8)
                tmem_st_32x32b_x8(tmem_acc + bz * NP + col0 + c0 + lanes, zero);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(acce0);
            mbar_arrive(acce0 + 8u);
        }
        pdl_wait();   // C is zeroed by the prologue just before
        uint32_t ch = 0;
        Cursor c = cursor_at(p, lo);
        for (int64_t i = lo; i < hi; ++i, c.advance(p.num_sb)) {
            if (!chunk_ends(p, c, i + 1 == hi)) continue;
            const uint32_t buf = ch & 1u, aph = (ch >> 1) & 1u;
            int got = 1;
            if (lane == 0) got = wait_bounded(accf0 + 8u * buf, aph, abort_flag, p.err, kDevErrTimeoutEpilogue);
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) break;
            tc_fence_after();
            const uint32_t taddr = tmem_acc + buf * NP + col0 + lanes;
            // the whole chunk into registers (one wait), the accumulator
            // zeroed and released at once, and only then the atomics into C,
            // so the MMAs into this accumulator never wait for them
            uint32_t v[Cfg::EPI_COLS / 8][8];
#pragma unroll
            for (int g8 = 0; g8 < Cfg::EPI_COLS / 8; ++g8) tmem_ld_32x32b_x8(taddr + g8 * 8, v[g8]);
            tmem_wait_ld();
#pragma unroll
            for (int g8 = 0; g8 < Cfg::EPI_COLS / 8; ++g8) tmem_st_32x32b_x8(taddr + g8 * 8, zero);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce0 + 8u * buf);
            const int64_t j = static_cast<int64_t>(c.tile) * 128 + jrow;
            if (j < p.n) {
                int32_t* out = p.C + static_cast<int64_t>(col0) * p.n + j;
#pragma unroll
                for (int g8 = 0; g8 < Cfg::EPI_COLS / 8; ++g8)
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc)
                        if (g8 * 8 + cc < rows)
                            atomicAdd(out + static_cast<int64_t>(g8 * 8 + cc) * p.n,
                                      __float2int_rn(__uint_as_float(v[g8][cc])));   // exact
            }
            ++ch;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

template <int NP>
cudaError_t launch_np(const int8_t* Bt, const uint16_t* A16, int32_t* C, int* err, int64_t m, int64_t n, int64_t k,
                      int num_sms, cudaStream_t stream) {
    using Cfg = SkCfg<NP>;
    auto enc = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
    if (!enc) return cudaErrorInvalidValue;
    CUtensorMap mB, mA;
    {
        // int8 Bt: 128-byte x 128-row boxes, 128-byte swizzle; K and rows
        // beyond the matrix read as zero
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(n)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(k)};
        cuuint32_t box[2] = {128u, 128u};
        cuuint32_t estr[2] = {1u, 1u};
        if (enc(&mB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(Bt), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // f16 activations: 64 K x NP rows per box (rows >= m read as zero)
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(m)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(k) * 2u};
        cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(NP)};
        cuuint32_t estr[2] = {1u, 1u};
        if (enc(&mA, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t*>(A16), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    SkParams p;
    p.C = C;
    p.err = err;
    p.m = static_cast<int>(m);
    p.n = static_cast<int>(n);
    p.num_sb = static_cast<int>((k + 255) / 256);
    p.tiles = static_cast<int>((n + 127) / 128);
    p.iters = static_cast<int64_t>(p.tiles) * p.num_sb;
    int64_t grid = num_sms;
    if (grid > p.iters) grid = p.iters;
    p.iters32 = (p.iters * (grid + 1)) < (int64_t(1) << 32) ? 1 : 0;
    auto kern = skinny_tc_kernel<NP>;
    cudaError_t e = kernel_attrs_once(reinterpret_cast<const void*>(kern), static_cast<int>(Cfg::SMEM), false);
    if (e != cudaSuccess) return e;
    // Programmatic dependent launch: the kernel may start while the prologue
    // before it (and, through it, the previous call's kernel) still runs.
    // Until its grid dependency wait it only sets up; every load and every
    // write of C comes after.
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kSkThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, mB, mA, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

bool skinny_tc_supported(int64_t m, int64_t n, int64_t k, const void* A, const void* Bt) {
    return m >= 1 && m <= 128 && (k % 16) == 0 && n <= 2147483647LL - 128 &&
           ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(Bt)) & 15u) == 0;
}

cudaError_t launch_skinny_tc(const int8_t* Bt, const uint16_t* A16, int32_t* C, int* err, int64_t m, int64_t n,
                             int64_t k, int num_sms, cudaStream_t stream) {
    if (m <= 16) return launch_np<16>(Bt, A16, C, err, m, n, k, num_sms, stream);
    if (m <= 32) return launch_np<32>(Bt, A16, C, err, m, n, k, num_sms, stream);
    if (m <= 64) return launch_np<64>(Bt, A16, C, err, m, n, k, num_sms, stream);
    return launch_np<128>(Bt, A16, C, err, m, n, k, num_sms, stream);
}

}  // namespace gemm
