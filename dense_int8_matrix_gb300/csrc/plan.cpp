// Host tile selector: the five steps of patent CN114238853A
// ("一種矩陣乘分片配置選擇方法及系統"), re-derived for the sm_103a tensor core.
//
//   claim 1 step 1 / claim 2  enumerate tiles the matrix unit can run: BM in
//                             {64, 128} (M of one cta_group::1 MMA), BN in
//                             {32, 64, 128, 256} (multiples of the minimum
//                             N), plus the two-SM tile 256 x 256 (M of one
//                             cta_group::2 MMA, run by a pair of CTAs); K
//                             depth 64 16-bit elements per stage
//   claim 3                   drop tiles whose shared memory or TMEM (two
//                             accumulators of BN columns) exceed one SM
//   claim 4 S1-S3             Thread_Blocks = output tiles; keep tiles with at
//                             least one tile per SM; if none, the problem is
//                             too small: keep only the smallest tile
//   claim 5                   compute-to-memory ratio 2*BM*BN/((BM+BN)*2);
//                             keep the largest
//   claim 6                   block_per_cu from registers, shared memory and
//                             TMEM; waves = ceil(tiles/(SMs*block_per_cu));
//                             keep the fewest
//   (unstated tie-break)      larger BM*BN, then larger BM
//   claim 7                   every tile is a compiled template instance; the
//                             plan names the one to launch
//   (after step 5)            a multi-wave choice gives way to the two-SM
//                             tile when it covers C in one round of pairs and
//                             K has at least 12 steps
//   (after step 5, int8)      K split: small-MN, large-K problems whose choice
//                             runs in one wave take the two-SM tile split
//                             along K; otherwise the tail of a partial last
//                             round is split
// int8 problems with m <= 64, or m <= 128 and k % 16 == 0, are routed to the
// skinny path first.
#include <cstdint>

#include "../../include/dense_int8_matrix.h"
#include "internal.h"

namespace gemm {

namespace {

constexpr int64_t kSmemPerCtaMax = 232448;
constexpr int64_t kSmemPerSm = 233472;
constexpr int64_t kRegsPerSm = 65536;
constexpr int64_t kTmemColsPerSm = 512;
constexpr int64_t kMaxDim = 2147483647;
// Widen int8 A on chip in the two-SM kernel when C is at most this wide: the
// staged f16 copy of A costs 3 m*k bytes of traffic against 2 m*n*k flops.
constexpr int64_t kAOnChipMaxN = 512;
// The two-SM tile replaces a multi-wave one-SM choice only with at least this
// many K steps of 64.
constexpr int64_t kPairWaveMinKSteps = 12;

struct Tile {
    int bm, bn;
};
constexpr Tile kTiles[] = {{64, 32},  {64, 64},   {64, 128},  {64, 256}, {128, 32},
                           {128, 64}, {128, 128}, {128, 256}, {256, 256}};

bool is_pair(const Tile& t) { return t.bm == 256; }
int64_t tile_smem(const Tile& t) {
    return is_pair(t) ? static_cast<int64_t>(tc2_smem_bytes()) : static_cast<int64_t>(tc_smem_bytes(t.bm, t.bn));
}
// TMEM columns one CTA allocates: two accumulators of BN columns (the pair
// tile: 256 columns per accumulator in each CTA)
int64_t tile_tmem(const Tile& t) { return is_pair(t) ? 512 : tc_tmem_cols(t.bn); }
constexpr int kNumTiles = sizeof(kTiles) / sizeof(kTiles[0]);

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool tile_fits(const Tile& t) { return tile_smem(t) <= kSmemPerCtaMax && tile_tmem(t) <= kTmemColsPerSm; }

int64_t out_tiles(const Tile& t, int64_t m, int64_t n) { return ceil_div(m, t.bm) * ceil_div(n, t.bn); }
// Thread blocks (CTAs) of claim 4: two per tile for the pair tile.
int64_t out_ctas(const Tile& t, int64_t m, int64_t n) { return out_tiles(t, m, n) * (is_pair(t) ? 2 : 1); }

double tile_ratio(const Tile& t) {
    // flops of one K step over the bytes it stages: 2*BM*BN*BK / ((BM+BN)*BK*2)
    return 2.0 * t.bm * t.bn / ((t.bm + t.bn) * 2.0);
}

int tile_bpc(const Tile& t) {
    const int64_t by_regs = kRegsPerSm / (static_cast<int64_t>(kTcThreads) * tc_regs_per_thread(t.bn));
    const int64_t by_smem = kSmemPerSm / tile_smem(t);
    const int64_t by_tmem = kTmemColsPerSm / tile_tmem(t);
    int64_t b = by_regs;
    if (by_smem < b) b = by_smem;
    if (by_tmem < b) b = by_tmem;
    return static_cast<int>(b);
}

int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// After the tile and the K split: int8 problems on the two-SM tile with a
// narrow C and a 16-byte row pitch of int8 A widen A on chip; the workspace
// then holds only the f16 copy of Bt.
void set_a_on_chip(gemm_plan* p) {
    p->a_on_chip = (p->dtype == GEMM_DTYPE_I8 && p->bm == 256 && p->k % 16 == 0 && p->n <= kAOnChipMaxN) ? 1 : 0;
    if (p->a_on_chip) p->workspace_bytes = round_up(p->n * p->k_pitch * 2, 256);
}

}  // namespace

int tc_blocks_per_sm(int bm, int bn) { return tile_bpc(Tile{bm, bn}); }

gemm_status make_plan(int32_t dtype, int64_t m, int64_t k, int64_t n, int32_t num_sms, gemm_plan* out) {
    if (!out) return GEMM_ERR_INVALID_ARG;
    if (dtype != GEMM_DTYPE_I8 && dtype != GEMM_DTYPE_BF16) return GEMM_ERR_INVALID_ARG;
    if (m < 1 || k < 1 || n < 1 || m > kMaxDim || k > kMaxDim || n > kMaxDim) return GEMM_ERR_INVALID_ARG;
    if (num_sms < 1) return GEMM_ERR_INVALID_ARG;
    if (dtype == GEMM_DTYPE_I8 && k > GEMM_I8_MAX_K) return GEMM_ERR_OVERFLOW_RISK;

    gemm_plan p{};
    p.version = GEMM_PLAN_VERSION;
    p.dtype = dtype;
    p.num_sms = num_sms;
    p.m = m;
    p.k = k;
    p.n = n;

    // Routing: a skinny int8 problem streams Bt once, widening it to f16 on
    // chip; the tensor path would write and read an f16 copy of all of Bt.
    // Up to 128 rows when the skinny tensor-core kernel applies (k % 16 == 0).
    if (dtype == GEMM_DTYPE_I8 && (m <= 64 || (m <= 128 && k % 16 == 0))) {
        p.path = GEMM_PATH_SKINNY;
        p.bm = static_cast<int32_t>(m);
        p.bn = 32;
        p.bk = 16;
        p.stages = 1;
        const int64_t tiles = ceil_div(n, 32);
        if (tiles > kMaxDim) return GEMM_ERR_INVALID_ARG;
        p.tiles = static_cast<int32_t>(tiles);
        p.grid = p.tiles;
        p.bpc = 0;
        p.waves = 0;
        p.k_pitch = static_cast<int32_t>(k);
        p.chunk_k = static_cast<int32_t>(k);
        p.ratio = 2.0 * m / (m + 1.0);  // flops per byte streamed (m rows of A reused per Bt byte)
        p.workspace_bytes = 0;
        p.split_k = 1;
        p.split_from = p.tiles;
        *out = p;
        return GEMM_OK;
    }

    // Step 1: candidates; step 2: resource fit.
    bool alive[kNumTiles];
    for (int i = 0; i < kNumTiles; ++i) alive[i] = tile_fits(kTiles[i]);

    // Step 3: keep tiles that fill every SM with at least one output tile.
    bool any_full = false;
    for (int i = 0; i < kNumTiles; ++i)
        if (alive[i] && out_ctas(kTiles[i], m, n) >= num_sms) any_full = true;
    if (any_full) {
        for (int i = 0; i < kNumTiles; ++i)
            if (alive[i] && out_ctas(kTiles[i], m, n) < num_sms) alive[i] = false;
    } else {
        // Too small to fill the chip: only the smallest tile stays.
        int smallest = -1;
        for (int i = 0; i < kNumTiles; ++i) {
            if (!alive[i]) continue;
            if (smallest < 0) {
                smallest = i;
                continue;
            }
            const Tile& a = kTiles[i];
            const Tile& b = kTiles[smallest];
            const int64_t aa = static_cast<int64_t>(a.bm) * a.bn, bb = static_cast<int64_t>(b.bm) * b.bn;
            if (aa < bb || (aa == bb && a.bm < b.bm)) smallest = i;
        }
        for (int i = 0; i < kNumTiles; ++i) alive[i] = (i == smallest);
        p.fallback = 1;
    }

    // Step 4: largest compute-to-memory ratio.
    double best_ratio = -1.0;
    for (int i = 0; i < kNumTiles; ++i)
        if (alive[i] && tile_ratio(kTiles[i]) > best_ratio) best_ratio = tile_ratio(kTiles[i]);
    for (int i = 0; i < kNumTiles; ++i)
        if (alive[i] && tile_ratio(kTiles[i]) != best_ratio) alive[i] = false;

    // Step 5: fewest waves; then the tie-break.
    int best = -1;
    int64_t best_waves = 0;
    for (int i = 0; i < kNumTiles; ++i) {
        if (!alive[i]) continue;
        const Tile& t = kTiles[i];
        const int64_t w = ceil_div(out_ctas(t, m, n), static_cast<int64_t>(num_sms) * tile_bpc(t));
        bool take = false;
        if (best < 0 || w < best_waves) {
            take = true;
        } else if (w == best_waves) {
            const Tile& b = kTiles[best];
            const int64_t ta = static_cast<int64_t>(t.bm) * t.bn, tb = static_cast<int64_t>(b.bm) * b.bn;
            take = ta > tb || (ta == tb && t.bm > b.bm);
        }
        if (take) {
            best = i;
            best_waves = w;
        }
    }
    if (best < 0) return GEMM_ERR_INVALID_ARG;

    // Beyond the five steps (measured): a choice of two or more waves gives
    // way to the two-SM tile in one wave when that tile covers C in one round
    // of CTA pairs (step 3 rejected it for filling fewer than all SMs) and K
    // has at least kPairWaveMinKSteps steps.  Each SM then does the same
    // multiply-adds as in two waves of one-SM tiles, from half the staged
    // bytes per flop; with shorter K the two-SM tile's pipeline fill and
    // epilogue, which no second wave hides, cost more than that saves.
    {
        const int pair_idx = kNumTiles - 1;   // {256, 256}
        const Tile& pt = kTiles[pair_idx];
        const int64_t t2 = out_tiles(pt, m, n);
        if (best_waves >= 2 && !is_pair(kTiles[best]) && tile_fits(pt) && t2 <= num_sms / 2 &&
            ceil_div(k, kTcBK) >= kPairWaveMinKSteps) {
            best = pair_idx;
            best_waves = ceil_div(out_ctas(pt, m, n), static_cast<int64_t>(num_sms) * tile_bpc(pt));
        }
    }
    const Tile& t = kTiles[best];
    const int64_t tiles = out_tiles(t, m, n);
    if (tiles > kMaxDim) return GEMM_ERR_INVALID_ARG;
    const int bpc = tile_bpc(t);

    p.path = GEMM_PATH_TENSOR;
    p.bm = t.bm;
    p.bn = t.bn;
    p.bk = kTcBK;
    p.stages = kTcStages;
    p.tiles = static_cast<int32_t>(tiles);
    p.bpc = bpc;
    const int64_t slots = static_cast<int64_t>(num_sms) * bpc;
    if (is_pair(t)) {
        // CTAs in pairs: one pair per tile, at most one CTA per SM
        const int64_t pairs = slots / 2;
        p.grid = static_cast<int32_t>(2 * (tiles < pairs ? tiles : (pairs > 0 ? pairs : 1)));
    } else {
        p.grid = static_cast<int32_t>(tiles < slots ? tiles : slots);
    }
    p.waves = static_cast<int32_t>(best_waves);
    p.ratio = tile_ratio(t);
    // Staged 16-bit rows need a 16-byte pitch for TMA.
    const int64_t k_pitch = round_up(k, 8);
    if (k_pitch > kMaxDim) return GEMM_ERR_INVALID_ARG;
    p.k_pitch = static_cast<int32_t>(k_pitch);
    const int64_t num_kb = ceil_div(k, kTcBK);
    if (dtype == GEMM_DTYPE_I8) {
        p.chunk_k = kI8ChunkK;
        p.workspace_bytes = round_up(m * k_pitch * 2, 256) + round_up(n * k_pitch * 2, 256);
    } else {
        p.chunk_k = static_cast<int32_t>(num_kb * kTcBK > kMaxDim ? kMaxDim : num_kb * kTcBK);
        p.workspace_bytes = (k % 8 == 0) ? 0 : round_up(m * k_pitch * 2, 256) + round_up(n * k_pitch * 2, 256);
    }
    // Beyond the five steps, int8 only (the slices of an int8 product add
    // exactly):
    // (i) small-MN, large-K: a one-wave choice gives way to the two-SM tile
    //     split along K into S = min(pairs / its tiles, K steps / 16, 8)
    //     slices when S >= 2 (every slice at least one 1024-element chunk,
    //     all slices in one round);
    if (dtype == GEMM_DTYPE_I8 && best_waves == 1) {
        const Tile pair_tile{256, 256};
        const int64_t pairs = num_sms / 2;
        const int64_t t2 = out_tiles(pair_tile, m, n);
        int64_t s = t2 > 0 ? pairs / t2 : 0;
        if (s > num_kb / 16) s = num_kb / 16;
        if (s > kTcMaxSplit) s = kTcMaxSplit;
        if (s >= 2 && tile_fits(pair_tile) && t2 <= kMaxDim) {
            p.bm = 256;
            p.bn = 256;
            p.tiles = static_cast<int32_t>(t2);
            p.bpc = tile_bpc(pair_tile);
            p.grid = static_cast<int32_t>(2 * (t2 * s < pairs ? t2 * s : pairs));
            p.waves = static_cast<int32_t>(ceil_div(t2 * s, pairs));
            p.ratio = tile_ratio(pair_tile);
            p.split_k = static_cast<int32_t>(s);
            p.split_from = 0;
            set_a_on_chip(&p);
            *out = p;
            return GEMM_OK;
        }
    }
    // (ii) otherwise split the last, partial wave along K (over CTA pairs for
    //     the two-SM tile).
    const int64_t nchunks = ceil_div(num_kb, p.chunk_k / kTcBK);
    int64_t split_from = tiles;
    const int64_t workers = is_pair(t) ? p.grid / 2 : p.grid;
    p.split_k = tc_tail_split(tiles, workers, nchunks, dtype == GEMM_DTYPE_I8, &split_from);
    p.split_from = static_cast<int32_t>(split_from);
    set_a_on_chip(&p);
    *out = p;
    return GEMM_OK;
}

}  // namespace gemm
