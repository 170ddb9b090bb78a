"""Pins for the selector oracle: hand-worked examples of the patent's five
steps (tests/golden/selector_examples.txt, derivations in its header)."""

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
            d, m, k, n, sms, path, bm, bn, tiles, waves, fb = line.split()
            rows.append((d, int(m), int(k), int(n), int(sms), path, int(bm), int(bn),
                         int(tiles), int(waves), bool(int(fb))))
    return rows


EXAMPLES = load_examples()


@pytest.mark.parametrize("ex", EXAMPLES, ids=lambda e: "%s-%dx%dx%d-%d" % e[:5])
def test_selector_oracle_hand_examples(ex):
    d, m, k, n, sms, path, bm, bn, tiles, waves, fb = ex
    got = selector.select(d, m, k, n, sms)
    assert got["path"] == path
    if path == "tensor":
        assert (got["bm"], got["bn"]) == (bm, bn)
        assert got["tiles"] == tiles
        assert got["waves"] == waves
        assert got["fallback"] == fb


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
