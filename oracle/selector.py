"""Oracle for the tile-configuration selector (TEST INFRASTRUCTURE ONLY).

Only the tests may import it; the product's planner is separate C++ and
shares nothing with this file.  It has two parts, kept apart so that the
first can be checked against the patent alone:

1. ``five_steps`` restates the five-step method of patent CN114238853A
   ("一種矩陣乘分片配置選擇方法及系統", claim 1 steps 1-5 and claims 2-6), read
   for a GPU whose matrix unit is the sm_103a tensor core.  Besides the
   problem's (m, n) and the SM count, its inputs are the limits of one SM
   (``Sm``) and the resources each candidate kernel uses (``Candidate``):
   steps 2 and 5 take a kernel's registers, shared memory and threads as
   given, and the library's compiled kernels are one such table
   (``library_candidates``).
2. The library's own rules, which the pages do not contain: ``route`` sends
   small-m int8 problems to the skinny path before step 1; after step 5,
   ``pair_wave`` trades a multi-wave choice for the two-SM tile in one wave,
   ``k_split`` splits small-MN, large-K int8 problems along K, and
   ``a_on_chip`` says where int8 A is widened to f16.

``select`` composes them: route, the five steps, pair_wave, the K split,
a_on_chip.

Readings of the five steps (the patent's formulas did not survive
extraction):

Step 1 (claim 1 step 1, claim 2): the thread-block tiles the matrix unit
    can execute.  Tile sides are multiples of the unit's minimum shape
    ("TCUmin shape size"): BM in {64, 128} (the M of one tensor-core MMA
    issued by one CTA), BN in {32, 64, 128, 256}, and the 256 x 256 tile of
    the two-SM MMA (M = 256), run by a pair of thread blocks.
Step 2 (claim 3): drop tiles whose resources do not fit one SM: shared
    memory of a CTA above the per-CTA limit, or TMEM columns (two
    accumulators of BN columns) above the SM's.
Step 3 (claim 4 S1-S3): Thread_Blocks = the CTAs of the output tiling,
    ceil(m/BM) * ceil(n/BN) tiles times the CTAs per tile;
    min_theory_block_num = the SM count.  Keep tiles with Thread_Blocks >=
    min_theory_block_num.  If none qualifies the problem is too small to fill
    the chip; "set the reuse counts to 1" is read as: keep only the smallest
    tile.
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
"""

from __future__ import annotations

import math
from dataclasses import dataclass

BK_ELEMS = 64        # K elements of a 16-bit operand per pipeline stage (128 bytes)
ESIZE = 2            # bytes per staged operand element (int8 is staged as f16)


@dataclass(frozen=True)
class Sm:
    """Limits of one SM used by steps 2 and 5."""
    smem_per_cta_max: int = 232448   # bytes of shared memory one CTA may use
    smem_per_sm: int = 233472        # bytes of shared memory per SM
    regs_per_sm: int = 65536         # 32-bit registers per SM
    tmem_cols_per_sm: int = 512      # TMEM columns (each 128 lanes x 32 bit)


@dataclass(frozen=True)
class Candidate:
    """A candidate tile and the resources one CTA of its kernel uses."""
    bm: int
    bn: int
    threads: int
    regs_per_thread: int
    smem_bytes: int
    tmem_cols: int
    ctas_per_tile: int = 1


GB300_SM = Sm()


# ---------------------------------------------------------------------------
# The library's compiled kernels as step 1's candidates.  Every one-SM tile is
# a CTA of 384 threads with a 4-stage operand ring; registers per thread are
# what the kernel is compiled for (168 for the wide tiles, BN >= 128, whose
# epilogue keeps 64 or 128 running sums per thread; 80 for the narrow ones);
# shared memory is the ring + 1 KiB to align it to the 1024-byte swizzle atom
# + 1 KiB for barriers, plus 8 x 4 KiB of C staging on the wide BM = 128
# tiles; TMEM is two BN-column accumulators rounded up to a power of two
# (at least 32).  The two-SM tile: two CTAs per tile, each with a 6-stage ring
# of 128-row A and B halves, the C staging, and all 512 TMEM columns.

def _tmem_cols(bn: int) -> int:
    need = max(32, 2 * bn)
    cols = 32
    while cols < need:
        cols *= 2
    return cols


def library_candidates():
    out = []
    for bm in (64, 128):
        for bn in (32, 64, 128, 256):
            epilogue = 8 * 4096 if (bm == 128 and bn >= 128) else 0
            smem = 4 * (bm + bn) * BK_ELEMS * ESIZE + epilogue + 1024 + 1024
            out.append(Candidate(bm, bn, 384, 168 if bn >= 128 else 80, smem, _tmem_cols(bn)))
    out.append(Candidate(256, 256, 384, 168, 6 * (128 + 128) * BK_ELEMS * ESIZE + 8 * 4096 + 1024 + 1024,
                         512, ctas_per_tile=2))
    return out


# ---------------------------------------------------------------------------
# The five steps (patent claims 1-6), each a plain function.

def fits(c: Candidate, sm: Sm = GB300_SM) -> bool:
    """Step 2: the CTA's shared memory and TMEM fit one SM."""
    return c.smem_bytes <= sm.smem_per_cta_max and c.tmem_cols <= sm.tmem_cols_per_sm


def tiles(m: int, n: int, bm: int, bn: int) -> int:
    """Output tiles of the (m, n) result."""
    return math.ceil(m / bm) * math.ceil(n / bn)


def thread_blocks(m: int, n: int, c: Candidate) -> int:
    """Step 3's Thread_Blocks: CTAs over all output tiles."""
    return tiles(m, n, c.bm, c.bn) * c.ctas_per_tile


def ratio(bm: int, bn: int) -> float:
    """Step 4's compute-to-memory ratio (flops per staged byte)."""
    return 2.0 * bm * bn / ((bm + bn) * ESIZE)


def blocks_per_sm(c: Candidate, sm: Sm = GB300_SM) -> int:
    """Step 5's block_per_cu."""
    by_regs = sm.regs_per_sm // (c.threads * c.regs_per_thread)
    by_smem = sm.smem_per_sm // c.smem_bytes
    by_tmem = sm.tmem_cols_per_sm // c.tmem_cols
    return min(by_regs, by_smem, by_tmem)


def waves(m: int, n: int, c: Candidate, num_sms: int, sm: Sm = GB300_SM) -> int:
    """Step 5's Launch_kernel_times."""
    return math.ceil(thread_blocks(m, n, c) / (num_sms * blocks_per_sm(c, sm)))


def five_steps(m: int, n: int, num_sms: int, candidates=None, sm: Sm = GB300_SM) -> dict:
    """Patent CN114238853A claim 1 steps 1-5 for an m x n output on
    `num_sms` SMs; `candidates` defaults to the library's compiled kernels."""
    cands = list(candidates) if candidates is not None else library_candidates()   # step 1
    cands = [c for c in cands if fits(c, sm)]                                          # step 2
    filled = [c for c in cands if thread_blocks(m, n, c) >= num_sms]                  # step 3
    fallback = not filled
    cands = filled if filled else [min(cands, key=lambda c: (c.bm * c.bn, c.bm))]
    best_r = max(ratio(c.bm, c.bn) for c in cands)                                     # step 4
    cands = [c for c in cands if ratio(c.bm, c.bn) == best_r]
    best_w = min(waves(m, n, c, num_sms, sm) for c in cands)                           # step 5
    cands = [c for c in cands if waves(m, n, c, num_sms, sm) == best_w]
    cands.sort(key=lambda c: (c.bm * c.bn, c.bm), reverse=True)                        # tie-break
    c = cands[0]
    return {"bm": c.bm, "bn": c.bn, "tiles": tiles(m, n, c.bm, c.bn), "bpc": blocks_per_sm(c, sm),
            "waves": best_w, "fallback": fallback}


# ---------------------------------------------------------------------------
# The library's own rules around the five steps (not on the pages).

def route(dtype: str, m: int, k: int) -> str:
    """Before step 1: int8 problems with m <= 64, or m <= 128 when k is a
    multiple of 16, take the skinny path (Bt streamed once and widened on
    chip); every other problem takes the tensor-core path."""
    if dtype not in ("i8", "bf16"):
        raise ValueError(dtype)
    if dtype == "i8" and (m <= 64 or (m <= 128 and k % 16 == 0)):
        return "skinny"
    return "tensor"


PAIR_WAVE_MIN_K_STEPS = 12


def pair_wave(m: int, k: int, n: int, num_sms: int, chosen: dict) -> dict:
    """After step 5: when the five steps' choice needs two or more waves,
    while the two-SM tile (which step 3 rejects for filling fewer than all
    SMs) covers C in one round of CTA pairs (T2 = ceil(m/256) * ceil(n/256)
    <= floor(SMs / 2)) and K has at least 12 steps of 64 (ceil(k/64) >= 12),
    the two-SM tile replaces it: one wave, T2 tiles.  Each SM then does the
    same multiply-adds as in the two waves of one-SM tiles, from half the
    staged bytes per flop."""
    if chosen["waves"] < 2 or chosen["bm"] == 256:
        return chosen
    t2 = tiles(m, n, 256, 256)
    if t2 > num_sms // 2 or math.ceil(k / BK_ELEMS) < PAIR_WAVE_MIN_K_STEPS:
        return chosen
    pair = candidate(256, 256)
    return {"bm": 256, "bn": 256, "tiles": t2, "bpc": blocks_per_sm(pair),
            "waves": waves(m, n, pair, num_sms), "fallback": chosen["fallback"]}


def k_split(dtype: str, m: int, k: int, n: int, num_sms: int, chosen: dict) -> dict:
    """After step 5, int8 only (the slices of an int8 product add exactly):
    when the five steps' choice runs in one wave, the two-SM tile split into
    S slices along K replaces it if S = min(floor(pairs / T2),
    floor(k_steps / 16), 8) >= 2, with pairs = floor(SMs / 2), T2 =
    ceil(m/256) * ceil(n/256) and k_steps = ceil(k/64): every slice keeps at
    least one 1024-element chunk, and the slices of all tiles run at once.
    The plan then has T2 tiles, the two-SM tile's block_per_cu and
    ceil(T2 * S / pairs) = 1 wave; "fallback" still records step 3."""
    out = dict(chosen, split=1)
    if dtype != "i8" or chosen["waves"] != 1:
        return out
    pairs = num_sms // 2
    t2 = tiles(m, n, 256, 256)
    k_steps = math.ceil(k / BK_ELEMS)
    s = min(pairs // t2, k_steps // 16, 8)
    if s < 2:
        return out
    pair = [c for c in library_candidates() if c.ctas_per_tile == 2][0]
    return {"bm": 256, "bn": 256, "tiles": t2, "bpc": blocks_per_sm(pair), "waves": math.ceil(t2 * s / pairs),
            "fallback": chosen["fallback"], "split": s}


A_ON_CHIP_MAX_N = 512


def a_on_chip(dtype: str, k: int, n: int, chosen: dict) -> int:
    """After the K split: int8 problems on the two-SM tile with n <= 512 and k
    a multiple of 16 widen int8 A inside the GEMM instead of staging an f16
    copy (for a narrow C that copy moves more bytes than the multiply)."""
    return int(dtype == "i8" and chosen["bm"] == 256 and k % 16 == 0 and n <= A_ON_CHIP_MAX_N)


def select(dtype: str, m: int, k: int, n: int, num_sms: int) -> dict:
    """The whole selection the library's planner makes: route, the five
    steps, the pair-tile wave rule, the K split, where A is widened."""
    if route(dtype, m, k) == "skinny":
        return {"path": "skinny"}
    chosen = k_split(dtype, m, k, n, num_sms, pair_wave(m, k, n, num_sms, five_steps(m, n, num_sms)))
    return dict(chosen, path="tensor", a_on_chip=a_on_chip(dtype, k, n, chosen))


# Kept for the tests that look a candidate up by its tile.
def candidate(bm: int, bn: int) -> Candidate:
    for c in library_candidates():
        if (c.bm, c.bn) == (bm, bn):
            return c
    raise KeyError((bm, bn))
