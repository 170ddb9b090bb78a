"""Pins for the selector oracle, in two parts kept apart:

* the patent's five steps alone (``selector.five_steps``), against hand-worked
  examples on the library's candidate kernels and on a made-up candidate
  table (tests/golden/selector_five_steps.txt);
* the library's whole selection (``selector.select``: its routing, the five
  steps, its K split), against hand-worked examples
  (tests/golden/selector_library.txt).

Derivations are written out in each file's header."""

import os

import pytest

from oracle import selector

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# the made-up candidate table "toy" of selector_five_steps.txt
TOY = [
    selector.Candidate(64, 64, threads=128, regs_per_thread=64, smem_bytes=40000, tmem_cols=128),
    selector.Candidate(128, 128, threads=256, regs_per_thread=128, smem_bytes=100000, tmem_cols=512),
    selector.Candidate(128, 256, threads=256, regs_per_thread=200, smem_bytes=240000, tmem_cols=512),
    selector.Candidate(64, 128, threads=256, regs_per_thread=128, smem_bytes=60000, tmem_cols=600),
]
TABLES = {"lib": None, "toy": TOY}


def _rows(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def load_five_step_examples():
    return [(t, int(m), int(n), int(sms), int(bm), int(bn), int(tiles), int(waves), bool(int(fb)))
            for t, m, n, sms, bm, bn, tiles, waves, fb in _rows("selector_five_steps.txt")]


def load_examples():
    """The library's whole selection: (dtype, m, k, n, sms, path, bm, bn,
    tiles, waves, fallback, split)."""
    return [(d, int(m), int(k), int(n), int(sms), path, int(bm), int(bn), int(tiles), int(waves),
             bool(int(fb)), int(split))
            for d, m, k, n, sms, path, bm, bn, tiles, waves, fb, split in _rows("selector_library.txt")]


FIVE = load_five_step_examples()
EXAMPLES = load_examples()


@pytest.mark.parametrize("ex", FIVE, ids=lambda e: "%s-%dx%d-%d" % e[:4])
def test_five_steps_hand_examples(ex):
    table, m, n, sms, bm, bn, tiles, waves, fb = ex
    got = selector.five_steps(m, n, sms, TABLES[table])
    assert (got["bm"], got["bn"], got["tiles"], got["waves"], got["fallback"]) == (bm, bn, tiles, waves, fb)


@pytest.mark.parametrize("ex", EXAMPLES, ids=lambda e: "%s-%dx%dx%d-%d" % e[:5])
def test_library_selection_hand_examples(ex):
    d, m, k, n, sms, path, bm, bn, tiles, waves, fb, split = ex
    got = selector.select(d, m, k, n, sms)
    assert got["path"] == path
    if path == "tensor":
        assert (got["bm"], got["bn"]) == (bm, bn)
        assert got["tiles"] == tiles
        assert got["waves"] == waves
        assert got["fallback"] == fb
        assert got["split"] == split


def test_five_steps_do_not_depend_on_k_or_dtype():
    # the patent's steps see only the output tiling: k and the dtype enter
    # through the library's rules alone, none of which applies with 8 K steps
    for m, n in [(1000, 3000), (4097, 255), (8192, 8192), (2048, 2048)]:
        for d in ("bf16", "i8"):
            a = selector.select(d, m, 512, n, 148)
            b = selector.five_steps(m, n, 148)
            assert (a["bm"], a["bn"], a["tiles"], a["waves"]) == (b["bm"], b["bn"], b["tiles"], b["waves"])


def test_pair_wave_rule():
    # a multi-wave one-SM choice gives way to the two-SM tile in one wave only
    # when T2 fits one round of pairs and K has at least 12 steps
    assert selector.select("i8", 1000, 777, 3000, 148)["bm"] == 256
    assert selector.select("i8", 1000, 704, 3000, 148)["bm"] == 128      # 11 K steps
    # step 3 rejects the two-SM tile exactly when its CTAs (2 T2) are fewer
    # than the SMs, i.e. when it fits one round of pairs; a larger problem
    # keeps the five steps' own two-SM choice, in two waves
    got = selector.select("i8", 2500, 4096, 3000, 148)
    assert (got["bm"], got["tiles"], got["waves"]) == (256, 120, 2)
    got = selector.select("bf16", 3000, 1000, 1000, 152)
    assert (got["bm"], got["tiles"], got["waves"]) == (256, 48, 1)


def test_ratio_closed_form():
    # TLP of a square tile BM = BN = b with 2-byte elements is b / 2
    for b in (64, 128, 256):
        assert selector.ratio(b, b) == b / 2
    # the library's shared-memory sizes: ring of (BM + BN) * 128 bytes per stage
    assert selector.candidate(128, 256).smem_bytes == 4 * 384 * 128 + 8 * 4096 + 2048
    assert selector.candidate(64, 256).smem_bytes == 4 * 320 * 128 + 2048


def test_every_library_candidate_fits_and_the_toy_table_drops_two():
    assert all(selector.fits(c) for c in selector.library_candidates())
    assert len(selector.library_candidates()) == 9
    assert [selector.fits(c) for c in TOY] == [True, True, False, False]


def test_routing_is_the_librarys_rule():
    assert selector.route("i8", 64, 7) == "skinny"
    assert selector.route("i8", 128, 8192) == "skinny"
    assert selector.route("i8", 128, 8190) == "tensor"
    assert selector.route("i8", 129, 8192) == "tensor"
    assert selector.route("bf16", 1, 8192) == "tensor"


def test_k_split_only_for_int8_one_wave_long_k():
    # the K split never applies to bf16, to multi-wave choices, or when a
    # slice would hold fewer than 16 K steps
    assert selector.select("bf16", 1024, 16384, 1024, 148)["split"] == 1
    assert selector.select("i8", 4096, 16384, 4096, 148)["split"] == 1
    assert selector.select("i8", 512, 1023, 512, 148)["split"] == 1    # 15 K steps
    assert selector.select("i8", 512, 2048, 512, 148)["split"] == 2    # 32 K steps
    # the slices of all tiles fit one round of pairs
    for shape in [(512, 8192, 512), (4097, 16384, 255), (1024, 16384, 1024), (300, 65536, 300)]:
        got = selector.select("i8", *shape, 148)
        assert got["split"] >= 2 and got["tiles"] * got["split"] <= 74 and got["waves"] == 1


@pytest.mark.parametrize("mistake", ["ratio_uses_bm_twice", "step3_counts_tiles_not_ctas",
                                     "step5_ignores_tmem", "tie_break_smaller_first"])
def test_a_planted_mistake_fails_a_hand_example(monkeypatch, mistake):
    # each plausible slip in the five steps changes at least one hand-worked
    # result, so the examples would catch it
    if mistake == "ratio_uses_bm_twice":
        monkeypatch.setattr(selector, "ratio", lambda bm, bn: 2.0 * bm * bm / ((bm + bm) * 2))
    elif mistake == "step3_counts_tiles_not_ctas":
        monkeypatch.setattr(selector, "thread_blocks", lambda m, n, c: selector.tiles(m, n, c.bm, c.bn))
    elif mistake == "step5_ignores_tmem":
        def bpc(c, sm=selector.GB300_SM):
            return min(sm.regs_per_sm // (c.threads * c.regs_per_thread), sm.smem_per_sm // c.smem_bytes)
        monkeypatch.setattr(selector, "blocks_per_sm", bpc)
    elif mistake == "tie_break_smaller_first":
        real = selector.five_steps

        def five(m, n, sms, candidates=None, sm=selector.GB300_SM):
            cands = list(candidates) if candidates is not None else selector.library_candidates()
            out = real(m, n, sms, cands, sm)
            # pick the smallest among the equal-wave, equal-ratio tiles instead
            ties = [c for c in cands if selector.fits(c, sm)
                    and selector.ratio(c.bm, c.bn) == selector.ratio(out["bm"], out["bn"])
                    and selector.thread_blocks(m, n, c) >= sms]
            if len(ties) > 1:
                c = min(ties, key=lambda c: (c.bm * c.bn, c.bm))
                out = dict(out, bm=c.bm, bn=c.bn, tiles=selector.tiles(m, n, c.bm, c.bn))
            return out
        monkeypatch.setattr(selector, "five_steps", five)
    failures = 0
    for table, m, n, sms, bm, bn, tiles, waves, fb in FIVE:
        got = selector.five_steps(m, n, sms, TABLES[table])
        if (got["bm"], got["bn"], got["tiles"], got["waves"], got["fallback"]) != (bm, bn, tiles, waves, fb):
            failures += 1
    assert failures >= 1
