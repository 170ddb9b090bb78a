"""Pins for the selector oracle: hand-worked examples of the patent's five
steps and of the K split after them (tests/golden/selector_examples.txt,
derivations in its header)."""

import os

import pytest

from oracle import selector

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "selector_examples.txt")


def load_examples():
    rows = []
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            d, m, k, n, sms, path, bm, bn, tiles, waves, fb, split = line.split()
            rows.append((d, int(m), int(k), int(n), int(sms), path, int(bm), int(bn),
                         int(tiles), int(waves), bool(int(fb)), int(split)))
    return rows


EXAMPLES = load_examples()


@pytest.mark.parametrize("ex", EXAMPLES, ids=lambda e: "%s-%dx%dx%d-%d" % e[:5])
def test_selector_oracle_hand_examples(ex):
    d, m, k, n, sms, path, bm, bn, tiles, waves, fb, split = ex
    got = selector.select(d, m, k, n, sms)
    assert got["path"] == path
    if path == "tensor":
        assert (got["bm"], got["bn"]) == (bm, bn)
        assert got["tiles"] == tiles
        assert got["waves"] == waves
        assert got["fallback"] == fb
        assert got["split"] == split


def test_selector_ratio_closed_form():
    # TLP of a square tile BM = BN = b with 2-byte elements is b / 2.
    for b in (64, 128):
        assert selector.ratio(b, b) == b / 2
    # the traffic of a (BM, BN) tile per K step is (BM + BN) * BK * 2 bytes
    assert selector.smem_per_cta(128, 256) == 4 * 384 * 128 + 8 * 4096 + 2048
    assert selector.smem_per_cta(64, 256) == 4 * 320 * 128 + 2048


def test_every_candidate_fits():
    assert all(selector.fits(*c) for c in selector.candidates())
    assert len(selector.candidates()) == 9


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
