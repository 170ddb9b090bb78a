"""GPU parity of the requantising entry point, gemm_i8_run_requant, through
the C ABI: D = q((float(C) * row_scale) * col_scale) with q = bfloat16 or
saturated int8, bit-exact against the CPU oracle (oracle.requant applied to
oracle.gemm_i8).  Covers the epilogue-fused path (whole tiles of both tensor
kernels), the scratch path (K-split tiles, the skinny path), ragged shapes,
unaligned outputs and special scales."""

import numpy as np
import pytest
import torch

import oracle
from dense_int8_matrix_gb300 import binding as B
from dense_int8_matrix_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_int8_matrix_gb300 import build
    build.build()
    oracle.build()
    B.load()
    yield
    st, code = B.gemm_device_error()
    assert st == B.GEMM_OK, "device error word set: code %d" % code


def _bits16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def gpu_requant(A, Bt, rs, cs, out, plan=None, d_offset=0, poison=True):
    """D from the GPU (CPU tensor: bfloat16 bits as uint16, or int8); the D
    buffer starts `d_offset` elements into a larger poisoned allocation."""
    m, k = A.shape
    n = Bt.shape[0]
    if plan is None:
        plan = B.gemm_i8_plan(m, k, n)
    dt = torch.bfloat16 if out == "bf16" else torch.int8
    buf = torch.empty(m * n + d_offset + 64, dtype=dt, device="cuda")
    if poison:
        buf.view(torch.int16 if out == "bf16" else torch.int8).fill_(0x5A5A if out == "bf16" else 0x5A)
    D = buf[d_offset:d_offset + m * n].view(m, n)
    B.gemm_i8_run_requant(plan, A.cuda(), Bt.cuda(), rs.cuda(), cs.cuda(), D.data_ptr(),
                          out_type=B.GEMM_OUT_BF16 if out == "bf16" else B.GEMM_OUT_I8)
    torch.cuda.synchronize()
    tail = buf[d_offset + m * n:].cpu()
    assert bool((tail.view(torch.int16 if out == "bf16" else torch.int8)
                 == (0x5A5A if out == "bf16" else 0x5A)).all()) or not poison, "write past the end of D"
    D = D.cpu()
    return _bits16(D) if out == "bf16" else D.numpy()


def assert_requant_exact(A, Bt, rs, cs, out, got):
    C = oracle.gemm_i8(A.numpy(), Bt.numpy())
    want = oracle.requant(C, rs.numpy(), cs.numpy(), out)
    if out == "bf16":
        nan_g = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
        nan_w = ((want & 0x7F80) == 0x7F80) & ((want & 0x7F) != 0)
        assert np.array_equal(nan_g, nan_w), "NaN positions differ"
        got = np.where(nan_g, 0, got)
        want = np.where(nan_w, 0, want)
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        i, j = bad[0]
        raise AssertionError("%d of %d elements differ; first at (%d, %d): gpu %r oracle %r (C %d)"
                             % (len(bad), got.size, i, j, got[i, j], want[i, j], C[i, j]))


def _case(m, k, n, seed, kind="uniform"):
    if kind == "skinny":
        A, Bt = workloads.make_inputs("i8_skinny", (m, k, n))
        rs, cs = workloads.requant_scales(m, n, k, seed, c_std_per_sqrt_k=(1365.0 * 1024.0) ** 0.5)
    else:
        A = workloads.random_i8((m, k), seed)
        Bt = workloads.random_i8((n, k), seed + 1)
        rs, cs = workloads.requant_scales(m, n, k, seed + 2)
    return A, Bt, rs, cs


@pytest.mark.parametrize("out", ["bf16", "i8"])
@pytest.mark.parametrize("m,k,n", [(1000, 777, 3000), (4096, 4096, 4096), (4097, 16384, 255), (300, 2100, 700)])
def test_requant_planned_shapes(m, k, n, out):
    # (1000,777,3000): whole one-SM tiles; 4096^3: two-SM tiles with a split
    # tail (fused + scratch); (4097,16384,255): every tile split along K
    A, Bt, rs, cs = _case(m, k, n, 7 + m)
    assert_requant_exact(A, Bt, rs, cs, out, gpu_requant(A, Bt, rs, cs, out))


@pytest.mark.parametrize("out", ["bf16", "i8"])
@pytest.mark.parametrize("m", [1, 16, 64, 128])
def test_requant_skinny(m, out):
    A, Bt, rs, cs = _case(m, 8192, 8192, 30 + m, "skinny")
    assert_requant_exact(A, Bt, rs, cs, out, gpu_requant(A, Bt, rs, cs, out))


def test_requant_skinny_cuda_core_path():
    # k % 16 != 0: the CUDA-core skinny kernel fills the int32 scratch
    A, Bt, rs, cs = _case(8, 1000, 777, 50)
    for out in ("bf16", "i8"):
        assert_requant_exact(A, Bt, rs, cs, out, gpu_requant(A, Bt, rs, cs, out))


TILES = [(bm, bn) for bm in (64, 128) for bn in (32, 64, 128, 256)] + [(256, 256)]


@pytest.mark.parametrize("bm,bn", TILES)
@pytest.mark.parametrize("grid,split", [(5, 1), (1000, 3)])
def test_requant_every_tile(bm, bn, grid, split):
    # every compiled tile fused (split 1) and through the scratch path (every
    # tile split 3 ways); ragged m and n
    m, k, n = 300, 2100, 700
    A, Bt, rs, cs = _case(m, k, n, 60)
    p = B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, m, k, n, torch.cuda.get_device_properties(0).multi_processor_count)
    p.bm, p.bn = bm, bn
    p.grid = grid if bm != 256 else 2 * max(1, grid // 2)
    if split > 1:
        p.split_k, p.split_from = split, 0
    else:
        p.split_k, p.split_from = 1, max(1, p.tiles)
    for out in ("bf16", "i8"):
        assert_requant_exact(A, Bt, rs, cs, out, gpu_requant(A, Bt, rs, cs, out, plan=p))


@pytest.mark.parametrize("m,k,n", [(257, 1024, 1001), (130, 64, 9), (513, 520, 255), (200, 4096, 4096)])
@pytest.mark.parametrize("d_offset", [0, 1])
def test_requant_ragged_and_unaligned_output(m, k, n, d_offset):
    # n % 8 != 0 and D one element off its alignment: the scalar store path
    A, Bt, rs, cs = _case(m, k, n, 70 + n)
    for out in ("bf16", "i8"):
        assert_requant_exact(A, Bt, rs, cs, out, gpu_requant(A, Bt, rs, cs, out, d_offset=d_offset))


def test_requant_special_scales():
    # zero, negative and huge scales: infinities, NaN (infinity times zero),
    # saturation of both signs
    m, k, n = 256, 1024, 512
    A = workloads.random_i8((m, k), 90)
    Bt = workloads.random_i8((n, k), 91)
    rs = torch.ones(m, dtype=torch.float32)
    cs = torch.ones(n, dtype=torch.float32)
    rs[0], rs[1], rs[2], rs[3] = 0.0, -1.0, 3.0e38, -3.0e38
    cs[0], cs[1], cs[2], cs[3] = 0.0, -2.0, 1.0e-30, 1.0e30
    for out in ("bf16", "i8"):
        assert_requant_exact(A, Bt, rs, cs, out, gpu_requant(A, Bt, rs, cs, out))


def test_requant_twice_in_a_row_matches_int32_path():
    # two calls in a row into the same D give the same result, and q of
    # gemm_i8_run's int32 C (through the oracle's q) equals the fused output
    m, k, n = 2048, 3072, 2560
    A, Bt, rs, cs = _case(m, k, n, 95)
    plan = B.gemm_i8_plan(m, k, n)
    C = torch.empty((m, n), dtype=torch.int32, device="cuda")
    B.gemm_i8_run(plan, A.cuda(), Bt.cuda(), C)
    torch.cuda.synchronize()
    for out in ("bf16", "i8"):
        want = oracle.requant(C.cpu().numpy(), rs.numpy(), cs.numpy(), out)
        first = gpu_requant(A, Bt, rs, cs, out, plan=plan)
        second = gpu_requant(A, Bt, rs, cs, out, plan=plan, poison=False)
        assert np.array_equal(first, want) and np.array_equal(second, want)


def test_requant_rejects_bad_arguments():
    import ctypes
    lib = B.load()
    plan = B.gemm_i8_plan(256, 256, 256)
    buf = torch.zeros(1 << 20, dtype=torch.int8, device="cuda")
    p = buf.data_ptr()
    st = lib.gemm_i8_run_requant(ctypes.byref(plan), p, p, p, p, 3, p, None)
    assert st == B.GEMM_ERR_INVALID_ARG
    st = lib.gemm_i8_run_requant(ctypes.byref(plan), p, p, p + 4, p, B.GEMM_OUT_I8, p, None)
    assert st == B.GEMM_ERR_MISALIGNED
    st = lib.gemm_i8_run_requant(ctypes.byref(plan), p, p, p, p, B.GEMM_OUT_BF16, p + 1, None)
    assert st == B.GEMM_ERR_MISALIGNED
    st = lib.gemm_i8_run_requant(ctypes.byref(plan), p, p, None, p, B.GEMM_OUT_I8, p, None)
    assert st == B.GEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("m,k,n", [(4097, 16384, 255), (1000, 4096, 512), (10240, 1024, 256)])
def test_requant_with_a_widened_on_chip(m, k, n):
    # plans that widen int8 A inside the two-SM kernel (a_on_chip = 1), with
    # every tile split along K (the scratch path) or, for (10240, 1024, 256),
    # whole tiles (40 tiles in one wave: requantised in the epilogue)
    A, Bt, rs, cs = _case(m, k, n, 110 + n)
    plan = B.gemm_i8_plan(m, k, n)
    assert plan.a_on_chip == 1
    for out in ("bf16", "i8"):
        assert_requant_exact(A, Bt, rs, cs, out, gpu_requant(A, Bt, rs, cs, out, plan=plan))
