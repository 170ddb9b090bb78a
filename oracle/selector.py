"""Oracle for the tile-configuration selector (TEST INFRASTRUCTURE ONLY).

A plain, step-by-step restatement of the five-step method of patent
CN114238853A ("一種矩陣乘分片配置選擇方法及系統", claim 1 steps 1-5 and claims
2-6), read for a GPU whose matrix unit is the sm_103a tensor core.  Only the
tests may import it; the product's planner is separate C++ and shares nothing
with this file.

The patent's formulas did not survive extraction, so each step states the
reading taken here:

Step 1 (claim 1 step 1, claim 2): enumerate the thread-block tiles that the
    matrix unit can execute.  Tile sides are multiples of the unit's minimum
    shape ("TCUmin shape size"): BM in {64, 128} (the M of one tensor-core MMA
    issued by one CTA) and BN in {32, 64, 128, 256}; and the 256 x 256 tile of
    the two-SM MMA (M = 256), which a pair of thread blocks runs, each with
    the resources of a (128, 256)-sized CTA.  The K depth of a stage is BK =
    64 elements of a 16-bit operand (128 bytes, one swizzle row).
Step 2 (claim 3): drop tiles whose resources do not fit one SM: shared memory
    of the CTA above the per-CTA limit, or a TMEM accumulator (two buffers of
    BN columns) above the 512 columns of an SM.
Step 3 (claim 4 S1-S3): Thread_Blocks = ceil(m/BM) * ceil(n/BN) (the output
    tiles), twice that for the two-SM tile (two thread blocks per tile);
    min_theory_block_num = the SM count.  Keep tiles with
    Thread_Blocks >= min_theory_block_num.  If none qualifies the problem is
    too small to fill the chip; "set the reuse counts to 1" is read as: keep
    only the smallest tile, (64, 32).
Step 4 (claim 5): compute-to-memory ratio of one K step,
    TLP = 2*BM*BN*BK / ((BM + BN)*BK*esize) = 2*BM*BN / ((BM + BN)*esize),
    with the right-matrix tile read as (BK, BN) (the claim's second
    "m_tiles" taken as n_tiles) and esize = 2 bytes (both dtypes are staged
    as 16-bit operands).  Keep every tile with the largest TLP.
Step 5 (claim 6): block_per_cu = min(registers of an SM // registers of a
    CTA, shared memory of an SM // shared memory of a CTA, TMEM columns of an
    SM // TMEM columns of a CTA); Launch_kernel_times (waves) =
    ceil(Thread_Blocks / (SMs * block_per_cu)).  Keep the fewest waves.
Tie-break (the pages are silent): larger BM*BN, then larger BM.
Routing (before step 1, the library's own rule): int8 problems with m <= 64,
or m <= 128 when k is a multiple of 16, go to the skinny path.
K split (after step 5, the library's rule for small-MN, large-K problems,
    where the pages' split-K technique applies: int8 only, since the slices
    of an int8 product add exactly): when the five steps' choice runs in one
    wave, the two-SM tile split into S slices along K replaces it if
    S = min(floor(pairs / T2), floor(k_steps / 16), 8) >= 2, with pairs =
    floor(SMs / 2), T2 = ceil(m/256) * ceil(n/256) and k_steps = ceil(k/64):
    every slice keeps at least one 1024-element chunk, and the slices of all
    tiles run at once.  The plan then has T2 tiles, block_per_cu 1 and
    ceil(T2 * S / pairs) = 1 wave; "fallback" still records step 3.
"""

from __future__ import annotations

import math

# Hardware characteristics of one GB300 SM used by steps 2 and 5.
SMEM_PER_CTA_MAX = 232448       # bytes of shared memory one CTA may use
SMEM_PER_SM = 233472            # bytes of shared memory per SM
REGS_PER_SM = 65536             # 32-bit registers per SM
TMEM_COLS_PER_SM = 512          # TMEM columns (each 128 lanes x 32 bit)

# The candidate kernels: every tile is a CTA of 384 threads with a 4-stage
# operand ring.  Register use per thread at launch is what the kernel is
# compiled for: 168 for the wide tiles (BN >= 128, whose epilogue keeps a
# 64- or 128-entry running sum per thread), 80 for the narrow ones.
STAGES = 4
BK_ELEMS = 64
ESIZE = 2
THREADS = 384


def regs_per_thread(bn: int) -> int:
    return 168 if bn >= 128 else 80


def is_pair(bm: int, bn: int) -> bool:
    return bm == 256


def smem_per_cta(bm: int, bn: int) -> int:
    # operand ring + 1 KiB for aligning the ring to the 1024-byte swizzle
    # atom + 1 KiB for barriers and bookkeeping; wide tiles (BM = 128,
    # BN >= 128) also stage C for TMA stores in 8 buffers of 4 KiB
    if is_pair(bm, bn):
        # each CTA of the pair: 6 stages of 128-row A and B halves
        return 6 * (128 + 128) * BK_ELEMS * ESIZE + 8 * 4096 + 1024 + 1024
    epilogue = 8 * 4096 if (bm == 128 and bn >= 128) else 0
    return STAGES * (bm + bn) * BK_ELEMS * ESIZE + epilogue + 1024 + 1024


def tmem_cols(bn: int) -> int:
    # two accumulators of BN columns per CTA (each CTA of a 256 x 256 pair
    # holds two of its 128 x 256 halves: 512 columns)
    need = max(32, 2 * bn)
    cols = 32
    while cols < need:
        cols *= 2
    return cols


def candidates():
    """Step 1: every (BM, BN) the tensor core can run as one CTA tile."""
    out = []
    for bm in (64, 128):
        for bn in (32, 64, 128, 256):
            out.append((bm, bn))
    out.append((256, 256))
    return out


def fits(bm: int, bn: int) -> bool:
    """Step 2: resource-fit filter."""
    if smem_per_cta(bm, bn) > SMEM_PER_CTA_MAX:
        return False
    if 2 * bn > TMEM_COLS_PER_SM:
        return False
    return True


def tiles(m: int, n: int, bm: int, bn: int) -> int:
    """Output tiles of the (m, n) result."""
    return math.ceil(m / bm) * math.ceil(n / bn)


def thread_blocks(m: int, n: int, bm: int, bn: int) -> int:
    """Step 3's Thread_Blocks: CTAs over all output tiles."""
    return tiles(m, n, bm, bn) * (2 if is_pair(bm, bn) else 1)


def ratio(bm: int, bn: int) -> float:
    """Step 4's compute-to-memory ratio (flops per staged byte)."""
    return 2.0 * bm * bn / ((bm + bn) * ESIZE)


def blocks_per_sm(bm: int, bn: int) -> int:
    """Step 5's block_per_cu."""
    by_regs = REGS_PER_SM // (THREADS * regs_per_thread(bn))
    by_smem = SMEM_PER_SM // smem_per_cta(bm, bn)
    by_tmem = TMEM_COLS_PER_SM // tmem_cols(bn)
    return min(by_regs, by_smem, by_tmem)


def waves(m: int, n: int, bm: int, bn: int, num_sms: int) -> int:
    """Step 5's Launch_kernel_times."""
    return math.ceil(thread_blocks(m, n, bm, bn) / (num_sms * blocks_per_sm(bm, bn)))


def select(dtype: str, m: int, k: int, n: int, num_sms: int) -> dict:
    """Run the routing and the five steps; return the chosen configuration."""
    if dtype not in ("i8", "bf16"):
        raise ValueError(dtype)
    if dtype == "i8" and (m <= 64 or (m <= 128 and k % 16 == 0)):
        return {"path": "skinny"}
    # step 1
    cands = candidates()
    # step 2
    cands = [c for c in cands if fits(*c)]
    # step 3
    filled = [c for c in cands if thread_blocks(m, n, *c) >= num_sms]
    fallback = not filled
    if fallback:
        cands = [min(cands, key=lambda c: (c[0] * c[1], c[0]))]
    else:
        cands = filled
    # step 4
    best_r = max(ratio(*c) for c in cands)
    cands = [c for c in cands if ratio(*c) == best_r]
    # step 5
    best_w = min(waves(m, n, *c, num_sms) for c in cands)
    cands = [c for c in cands if waves(m, n, *c, num_sms) == best_w]
    # tie-break
    cands.sort(key=lambda c: (c[0] * c[1], c[0]), reverse=True)
    bm, bn = cands[0]
    chosen = {
        "path": "tensor",
        "bm": bm,
        "bn": bn,
        "tiles": tiles(m, n, bm, bn),
        "bpc": blocks_per_sm(bm, bn),
        "waves": best_w,
        "fallback": fallback,
        "split": 1,
    }
    return k_split(dtype, m, k, n, num_sms, chosen)


def k_split(dtype: str, m: int, k: int, n: int, num_sms: int, chosen: dict) -> dict:
    """The K split after step 5 (see the module docstring)."""
    if dtype != "i8" or chosen["waves"] != 1:
        return chosen
    pairs = num_sms // 2
    t2 = tiles(m, n, 256, 256)
    k_steps = math.ceil(k / BK_ELEMS)
    s = min(pairs // t2, k_steps // 16, 8)
    if s < 2:
        return chosen
    return {
        "path": "tensor",
        "bm": 256,
        "bn": 256,
        "tiles": t2,
        "bpc": blocks_per_sm(256, 256),
        "waves": math.ceil(t2 * s / pairs),
        "fallback": chosen["fallback"],
        "split": s,
    }
