"""Host-side checks of the C ABI (no kernel launches): the library builds,
loads and exports every function include/dense_int8_matrix.h declares; the
planner matches the selector oracle; argument errors come back as statuses
before any CUDA call."""

import ctypes
import os
import random
import re

import pytest
import torch

from dense_int8_matrix_gb300 import binding as B
from dense_int8_matrix_gb300 import build as build_mod
from oracle import selector
from tests.test_selector_oracle import EXAMPLES

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dense_int8_matrix.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("gemm_i8_plan", "gemm_i8_run", "gemm_bf16_plan", "gemm_bf16_run",
                     "gemm_status_string"):
        assert required in names
    assert set(names) == set(B.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_exports_nothing_else(lib):
    """Internal C++ helpers stay hidden: the only defined text symbols in the
    dynamic table are the header's entry points."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", build_mod.LIB_PATH], check=True,
                         capture_output=True, text=True).stdout
    text_syms = sorted(line.split()[-1] for line in out.splitlines()
                       if len(line.split()) == 3 and line.split()[1] == "T")
    assert text_syms == declared_functions()


def test_plan_struct_layout(lib):
    # k = 700: 11 K steps, so the five steps' (128, 128) choice stands
    p = B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, 1000, 700, 3000, 148)
    assert ctypes.sizeof(B.gemm_plan) == 136
    assert (p.version, p.m, p.k, p.n) == (B.GEMM_PLAN_VERSION, 1000, 700, 3000)
    assert (p.bm, p.bn, p.tiles, p.waves, p.a_on_chip) == (128, 128, 192, 2, 0)
    assert p.k_pitch == 704 and p.chunk_k == 1024 and p.bk == 64 and p.stages == 4
    assert p.workspace_bytes == (1000 * 704 * 2 + 255) // 256 * 256 + (3000 * 704 * 2 + 255) // 256 * 256
    assert abs(p.ratio - 64.0) < 1e-12
    # the narrow shape widens A on chip: only the f16 copy of Bt is staged
    q = B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, 4097, 16384, 255, 148)
    assert (q.bm, q.a_on_chip, q.workspace_bytes) == (256, 1, 255 * 16384 * 2)


@pytest.mark.parametrize("ex", EXAMPLES, ids=lambda e: "%s-%dx%dx%d-%d" % e[:5])
def test_planner_hand_examples(lib, ex):
    d, m, k, n, sms, path, bm, bn, tiles, waves, fb, split = ex
    p = B.gemm_plan_for_sms(B.GEMM_DTYPE_I8 if d == "i8" else B.GEMM_DTYPE_BF16, m, k, n, sms)
    if path == "skinny":
        assert p.path == B.GEMM_PATH_SKINNY
        return
    assert p.path == B.GEMM_PATH_TENSOR
    assert (p.bm, p.bn, p.tiles, p.waves, bool(p.fallback)) == (bm, bn, tiles, waves, fb)
    if split > 1:   # every tile split along K
        assert (p.split_k, p.split_from) == (split, 0)
    else:           # at most the tail of a partial last round
        assert p.split_from > 0


def test_planner_matches_selector_oracle_sweep(lib):
    rng = random.Random(1234)
    dims = [1, 7, 63, 64, 65, 127, 128, 129, 200, 255, 256, 600, 777, 1000, 1536, 2048, 4095,
            4096, 4097, 8192, 12288, 16384, 30000]
    for _ in range(3000):
        d = rng.choice(["i8", "bf16"])
        m, k, n = rng.choice(dims), rng.choice(dims), rng.choice(dims)
        sms = rng.choice([1, 2, 64, 132, 148, 152, 160])
        if d == "i8" and k > B.GEMM_I8_MAX_K:
            continue
        want = selector.select(d, m, k, n, sms)
        p = B.gemm_plan_for_sms(B.GEMM_DTYPE_I8 if d == "i8" else B.GEMM_DTYPE_BF16, m, k, n, sms)
        if want["path"] == "skinny":
            assert p.path == B.GEMM_PATH_SKINNY
            continue
        got = (p.bm, p.bn, p.tiles, p.waves, p.bpc, bool(p.fallback), p.a_on_chip)
        assert got == (want["bm"], want["bn"], want["tiles"], want["waves"], want["bpc"],
                       want["fallback"], want["a_on_chip"]), (d, m, k, n, sms)
        if want["split"] > 1:   # every tile split: all slices in one round of pairs
            assert (p.split_k, p.split_from) == (want["split"], 0)
            assert p.grid == 2 * p.tiles * p.split_k <= 2 * (sms // 2)
        elif p.bm == 256:       # CTA pairs, one CTA per SM
            assert p.grid == 2 * min(p.tiles, max(1, sms // 2))
        else:
            assert p.grid == min(p.tiles, sms * p.bpc)


def test_plan_argument_errors(lib):
    p = B.gemm_plan()
    pl = ctypes.byref(p)
    assert lib.gemm_plan_for_sms(0, 0, 5, 5, 148, pl) == B.GEMM_ERR_INVALID_ARG
    assert lib.gemm_plan_for_sms(0, 5, -1, 5, 148, pl) == B.GEMM_ERR_INVALID_ARG
    assert lib.gemm_plan_for_sms(0, 5, 5, 2 ** 31, 148, pl) == B.GEMM_ERR_INVALID_ARG
    assert lib.gemm_plan_for_sms(7, 5, 5, 5, 148, pl) == B.GEMM_ERR_INVALID_ARG
    assert lib.gemm_plan_for_sms(0, 5, 5, 5, 0, pl) == B.GEMM_ERR_INVALID_ARG
    assert lib.gemm_plan_for_sms(0, 5, 5, 5, 148, None) == B.GEMM_ERR_INVALID_ARG
    assert lib.gemm_plan_for_sms(0, 128, 131072, 128, 148, pl) == B.GEMM_ERR_OVERFLOW_RISK
    assert lib.gemm_plan_for_sms(0, 128, 131071, 128, 148, pl) == B.GEMM_OK
    assert lib.gemm_plan_for_sms(1, 128, 1 << 20, 128, 148, pl) == B.GEMM_OK
    # the device planners reject bad arguments before touching the device
    assert lib.gemm_i8_plan(0, 5, 5, pl) == B.GEMM_ERR_INVALID_ARG
    assert lib.gemm_i8_plan(128, 200000, 128, pl) == B.GEMM_ERR_OVERFLOW_RISK
    assert lib.gemm_bf16_plan(5, 5, 5, None) == B.GEMM_ERR_INVALID_ARG


def test_run_argument_errors_before_any_launch(lib):
    p = B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, 256, 256, 256, 148)
    pl = ctypes.byref(p)
    s = None
    # null plan / pointers
    assert lib.gemm_i8_run(None, 4096, 4096, 4096, s) == B.GEMM_ERR_INVALID_ARG
    assert lib.gemm_i8_run(pl, None, 4096, 4096, s) == B.GEMM_ERR_INVALID_ARG
    assert lib.gemm_i8_run(pl, 4096, 4096, None, s) == B.GEMM_ERR_INVALID_ARG
    # misaligned operands
    assert lib.gemm_i8_run(pl, 4096 + 8, 4096, 4096, s) == B.GEMM_ERR_MISALIGNED
    assert lib.gemm_i8_run(pl, 4096, 4096 + 4, 4096, s) == B.GEMM_ERR_MISALIGNED
    assert lib.gemm_i8_run(pl, 4096, 4096, 4096 + 2, s) == B.GEMM_ERR_MISALIGNED
    # a plan of the other dtype or another version
    pb = B.gemm_plan_for_sms(B.GEMM_DTYPE_BF16, 256, 256, 256, 148)
    assert lib.gemm_i8_run(ctypes.byref(pb), 4096, 4096, 4096, s) == B.GEMM_ERR_INVALID_ARG
    assert lib.gemm_bf16_run(pl, 4096, 4096, 4096, s) == B.GEMM_ERR_INVALID_ARG
    bad = B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, 256, 256, 256, 148)
    bad.version = 99
    assert lib.gemm_i8_run(ctypes.byref(bad), 4096, 4096, 4096, s) == B.GEMM_ERR_INVALID_ARG
    bad = B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, 256, 256, 256, 148)
    bad.chunk_k = 2048   # would break the exactness bound of the int8 path
    assert lib.gemm_i8_run(ctypes.byref(bad), 4096, 4096, 4096, s) == B.GEMM_ERR_INVALID_ARG
    badb = B.gemm_plan_for_sms(B.GEMM_DTYPE_BF16, 256, 1000, 256, 148)
    badb.chunk_k = 512   # bf16 accumulates the whole K in one chunk
    assert lib.gemm_bf16_run(ctypes.byref(badb), 4096, 4096, 4096, s) == B.GEMM_ERR_INVALID_ARG
    bad = B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, 256, 256, 256, 148)
    bad.split_k = 9      # more K slices than the kernels take
    assert lib.gemm_i8_run(ctypes.byref(bad), 4096, 4096, 4096, s) == B.GEMM_ERR_INVALID_ARG
    bad = B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, 256, 256, 256, 148)
    bad.k_pitch = 100
    assert lib.gemm_i8_run(ctypes.byref(bad), 4096, 4096, 4096, s) == B.GEMM_ERR_INVALID_ARG
    # host forms check their arguments too
    assert lib.gemm_i8_run_host(None, 4096, 4096, 4096, s) == B.GEMM_ERR_INVALID_ARG
    assert lib.gemm_bf16_run_host(ctypes.byref(pb), None, 4096, 4096, s) == B.GEMM_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")
def test_no_device_means_error_not_fallback(lib):
    # With valid-looking arguments and no GPU, the call must fail with
    # GEMM_ERR_CUDA: there is no CPU path behind the ABI.
    p = B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, 256, 256, 256, 148)
    assert lib.gemm_i8_run(ctypes.byref(p), 4096, 4096, 4096, None) == B.GEMM_ERR_CUDA
    q = B.gemm_plan()
    assert lib.gemm_i8_plan(256, 256, 256, ctypes.byref(q)) == B.GEMM_ERR_CUDA
    code = ctypes.c_int32(0)
    assert lib.gemm_device_error(None, ctypes.byref(code)) == B.GEMM_ERR_CUDA


def test_status_strings(lib):
    for s, name in [(0, "GEMM_OK"), (2, "GEMM_ERR_MISALIGNED"), (5, "GEMM_ERR_OVERFLOW_RISK"),
                    (6, "GEMM_ERR_TIMEOUT")]:
        assert B.gemm_status_string(s) == name
    assert B.gemm_status_string(42) == "GEMM_ERR_UNKNOWN"


@pytest.mark.parametrize("m,k,n,sms,split,split_from", [
    (1536, 4096, 2048, 152, 3, 152),     # (128,128): 192 tiles = 152 + 40; 152 // 40 = 3
    (2048, 2048, 1536, 148, 2, 148),     # 192 = 148 + 44; 148 // 44 = 3, but only 2 K chunks
    (1024, 4096, 4096, 148, 1, 256),     # 256 = 148 + 108; 148 // 108 = 1: no split
    (1000, 777, 3000, 148, 1, 192),      # one K chunk: nothing to split
    (4096, 4096, 4096, 152, 2, 228),     # two-SM tile: 256 tiles = 3 * 76 pairs + 28; 76 // 28 = 2
    (8192, 8192, 8192, 152, 2, 988),     # two-SM tile: 1024 = 13 * 76 + 36; 76 // 36 = 2
    (2048, 1024, 2560, 148, 1, 80),      # two-SM tile: 80 tiles on 74 pairs, 74 // 6 = 12 but 1 K chunk
])
def test_tail_split_fields(lib, m, k, n, sms, split, split_from):
    p = B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, m, k, n, sms)
    tiles = p.tiles
    workers = p.grid // 2 if p.bm == 256 else p.grid   # CTA pairs for the two-SM tile
    full = (tiles // workers) * workers
    tail = tiles - full
    want = 1
    if tiles > workers and tail:
        nch = -(-(-(-k // 64)) // 16)
        want = min(workers // tail, nch, 8)
        if want < 2:
            want = 1
    assert p.split_k == want
    operands = (m * p.k_pitch * 2 + 255) // 256 * 256 + (n * p.k_pitch * 2 + 255) // 256 * 256
    assert p.workspace_bytes == operands   # the split needs no scratch: C is zeroed over its tiles
    if want > 1:
        assert (p.split_k, p.split_from) == (split, split_from)
        assert p.split_from + (tiles - p.split_from) * p.split_k <= full + workers
    else:
        assert p.split_from == tiles
    pb = B.gemm_plan_for_sms(B.GEMM_DTYPE_BF16, m, k, n, sms)
    assert pb.split_k == 1 and pb.split_from == pb.tiles


def test_skinny_plan_fields(lib):
    p = B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, 64, 8192, 8192, 148)
    assert p.path == B.GEMM_PATH_SKINNY and p.grid == 256 and p.workspace_bytes == 0
    p = B.gemm_plan_for_sms(B.GEMM_DTYPE_BF16, 64, 8192, 8192, 148)
    assert p.path == B.GEMM_PATH_TENSOR   # the skinny route is int8 only
    assert p.workspace_bytes == 0          # k % 8 == 0: bf16 operands are used in place
    p = B.gemm_plan_for_sms(B.GEMM_DTYPE_BF16, 64, 8190, 8192, 148)
    assert p.k_pitch == 8192 and p.workspace_bytes > 0
    # 64 < m <= 128: skinny only when the tensor-core skinny kernel applies
    assert B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, 128, 8192, 8192, 148).path == B.GEMM_PATH_SKINNY
    assert B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, 65, 16, 100, 148).path == B.GEMM_PATH_SKINNY
    assert B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, 128, 8200, 8192, 148).path == B.GEMM_PATH_TENSOR
    assert B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, 129, 8192, 8192, 148).path == B.GEMM_PATH_TENSOR
    assert B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, 64, 8190, 8192, 148).path == B.GEMM_PATH_SKINNY
