"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle.

int8 results must be bit-exact; bf16 results must satisfy
|C - oracle| <= 1e-3 * sum_k |a*b| elementwise.  Full comparisons at sizes
the oracle finishes in seconds and at the full 8192^3 sizes (the oracle's
row split over all host cores takes about 10 s for int8 there); the int8
8192^3 result is also checked by the Freivalds identity C r = A (B r), exact
in float64 at these magnitudes."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from dense_int8_matrix_gb300 import binding as B
from dense_int8_matrix_gb300 import workloads
from tests import gpu_util as G

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


# ------------------------------------------------------ named workloads ----

def test_workload_i8_256():
    A, Bt = workloads.make_inputs("i8_256", (256, 256, 256))
    G.assert_i8_exact(A, Bt, G.gpu_i8(A, Bt))


def test_workload_i8_4096():
    A, Bt = workloads.make_inputs("i8_4096", (4096, 4096, 4096))
    C = G.gpu_i8(A, Bt)
    G.assert_i8_exact(A, Bt, C)


@pytest.mark.parametrize("m", [1, 8, 16, 32, 64, 128])
def test_workload_i8_skinny(m):
    A, Bt = workloads.make_inputs("i8_skinny", (m, 8192, 8192))
    G.assert_i8_exact(A, Bt, G.gpu_i8(A, Bt))


@pytest.mark.parametrize("shape", [(1000, 777, 3000), (4097, 16384, 255)])
def test_workload_i8_ragged_full(shape):
    A, Bt = workloads.make_inputs("i8_ragged", shape)
    G.assert_i8_exact(A, Bt, G.gpu_i8(A, Bt))


def test_workload_i8_ragged_8192_full():
    # all 67,108,864 elements against the oracle, bit for bit, plus the
    # Freivalds identity as an independent check of both
    shape = (8192, 8192, 8192)
    A, Bt = workloads.make_inputs("i8_ragged", shape)
    C = G.gpu_i8(A, Bt)
    G.assert_i8_exact(A, Bt, C)
    G.freivalds_i8(A, Bt, C)


def test_workload_bf16_8192_full():
    # every element within |err| <= 1e-3 * sum_k |a*b| of the fp64 oracle
    shape = (8192, 8192, 8192)
    A, Bt = workloads.make_inputs("bf16_8192", shape)
    C = G.gpu_bf16(A, Bt)
    assert np.isfinite(C.numpy()).all()
    G.assert_bf16_close(A, Bt, C)


# -------------------------------------------------- every compiled tile ----

TILES = [(bm, bn) for bm in (64, 128) for bn in (32, 64, 128, 256)] + [(256, 256)]


def forced_plan(dtype, m, k, n, bm, bn, grid, split=1):
    # the planner's plan with another tile and grid; split > 1 splits every
    # tile into that many K slices, else the run decides (tail split only)
    p = B.gemm_plan_for_sms(dtype, m, k, n, torch.cuda.get_device_properties(0).multi_processor_count)
    p.bm, p.bn, p.grid = bm, bn, grid
    if split > 1:
        p.split_k, p.split_from = split, 0
    else:
        p.split_k, p.split_from = 1, max(1, p.tiles)
    return p


@pytest.mark.parametrize("bm,bn", TILES)
@pytest.mark.parametrize("grid,split", [(4, 1), (1000, 1), (1000, 3)])
def test_i8_every_tile(bm, bn, grid, split):
    # several tiles in both directions plus ragged tails; k = 2100 runs two
    # full 1024-element accumulator chunks and a ragged third one (or, split
    # 3 ways, slices of 11-11-11 K steps adding into C)
    m, k, n = 300, 2100, 700
    A = workloads.random_i8((m, k), 101)
    Bt = workloads.random_i8((n, k), 102)
    p = forced_plan(B.GEMM_DTYPE_I8, m, k, n, bm, bn, grid, split)
    C1 = G.gpu_i8(A, Bt, plan=p)
    G.assert_i8_exact(A, Bt, C1)
    if split > 1:
        assert torch.equal(C1, G.gpu_i8(A, Bt, plan=p))


@pytest.mark.parametrize("bm,bn", TILES)
def test_bf16_every_tile(bm, bn):
    m, k, n = 300, 1000, 700
    A = workloads.random_bf16((m, k), 103)
    Bt = workloads.random_bf16((n, k), 104)
    p = forced_plan(B.GEMM_DTYPE_BF16, m, k, n, bm, bn, 6)
    G.assert_bf16_close(A, Bt, G.gpu_bf16(A, Bt, plan=p))


# ------------------------------------------------------------ edge cases ----

@pytest.mark.parametrize("m,k,n", [
    (65, 1, 1), (65, 7, 3), (129, 63, 33), (200, 64, 64), (200, 65, 129),
    (130, 1024, 130), (130, 1025, 130), (257, 2048, 100), (300, 3073, 257),
    (1, 1, 1), (64, 16, 16), (63, 1000, 500), (8, 4100, 77), (2, 17, 5),
    (128, 8, 255), (513, 520, 1001),
])
def test_i8_edge_shapes(m, k, n):
    A = workloads.random_i8((m, k), m * 7 + k)
    Bt = workloads.random_i8((n, k), n * 11 + k)
    G.assert_i8_exact(A, Bt, G.gpu_i8(A, Bt))


@pytest.mark.parametrize("m,k,n", [(200, 1001, 300), (129, 8, 65), (65, 12, 40), (1, 64, 1)])
def test_bf16_edge_shapes(m, k, n):
    A = workloads.random_bf16((m, k), m + 3 * k)
    Bt = workloads.random_bf16((n, k), n + 5 * k)
    G.assert_bf16_close(A, Bt, G.gpu_bf16(A, Bt))


@pytest.mark.parametrize("m", [32, 200])
def test_i8_extreme_values_exact(m):
    # all -128: every fp32 chunk of 1024 products reaches exactly 2^24; the
    # int32 result 16384 * k is exact only if the chunked drain works
    k, n = 16384, 160
    A = torch.full((m, k), -128, dtype=torch.int8)
    Bt = torch.full((n, k), -128, dtype=torch.int8)
    C = G.gpu_i8(A, Bt)
    assert torch.all(C == 16384 * k)


def test_i8_max_k_exact():
    # k = 131071: the largest k the library accepts; C = 131071 * 16384
    m, k, n = 130, 131071, 40
    A = torch.full((m, k), -128, dtype=torch.int8)
    Bt = torch.full((n, k), -128, dtype=torch.int8)
    Bt[1::2] = 127
    C = G.gpu_i8(A, Bt)
    assert torch.all(C[:, 0::2] == 131071 * 16384)
    assert torch.all(C[:, 1::2] == -131071 * 16256)


def test_i8_alternating_signs_large_k():
    m, k, n = 256, 16384, 256
    A = workloads.random_i8((m, k), 5)
    sign = torch.where(torch.arange(k) % 2 == 0, 1, -1).to(torch.int8)
    A = torch.where(A == -128, torch.tensor(-127, dtype=torch.int8), A)
    Bt = (A[:n] * sign).to(torch.int8)
    G.assert_i8_exact(A, Bt, G.gpu_i8(A, Bt))


def test_bf16_integer_inputs_exact():
    # integer bf16 inputs with small sums: fp32 accumulation is exact
    m, k, n = 300, 2000, 260
    Ai = workloads.random_i8((m, k), 8, -16, 16)
    Bi = workloads.random_i8((n, k), 9, -16, 16)
    C = G.gpu_bf16(Ai.float().to(torch.bfloat16), Bi.float().to(torch.bfloat16))
    ref = oracle.gemm_i8(Ai.numpy(), Bi.numpy())
    assert np.array_equal(C.numpy(), ref.astype(np.float32))


# --------------------------------------------------------- ABI behaviour ----

def test_run_on_side_stream_and_repeat():
    m, k, n = 700, 3000, 500
    A = workloads.random_i8((m, k), 21)
    Bt = workloads.random_i8((n, k), 22)
    s = torch.cuda.Stream()
    dA, dB = A.cuda(), Bt.cuda()
    p = B.gemm_i8_plan(m, k, n)
    outs = []
    with torch.cuda.stream(s):
        for _ in range(3):
            C = torch.empty((m, n), dtype=torch.int32, device="cuda")
            B.gemm_i8_run(p, dA, dB, C, s)
            outs.append(C)
    s.synchronize()
    ref = oracle.gemm_i8(A.numpy(), Bt.numpy())
    for C in outs:
        assert np.array_equal(C.cpu().numpy(), ref)


def test_host_entry_points():
    m, k, n = 300, 1000, 200
    A = workloads.random_i8((m, k), 23)
    Bt = workloads.random_i8((n, k), 24)
    C = torch.empty((m, n), dtype=torch.int32).pin_memory()
    B.gemm_i8_run_host(B.gemm_i8_plan(m, k, n), A.pin_memory(), Bt.pin_memory(), C)
    G.assert_i8_exact(A, Bt, C)
    Ab = workloads.random_bf16((m, k), 25)
    Bb = workloads.random_bf16((n, k), 26)
    Cb = torch.empty((m, n), dtype=torch.float32)
    B.gemm_bf16_run_host(B.gemm_bf16_plan(m, k, n), Ab, Bb, Cb)
    G.assert_bf16_close(Ab, Bb, Cb)


@pytest.mark.parametrize("m,k,n,pinned", [(1, 8192, 8192, True), (16, 4096, 4096, False), (100, 2048, 1000, True),
                                           (8, 1000, 777, False)])
def test_host_entry_point_skinny(m, k, n, pinned):
    # skinny plans through the host-buffer form (copies in, prologue and
    # skinny kernel or the CUDA-core kernel, copy out), three calls in a row
    # into the same host C
    A = workloads.random_i8((m, k), 351 + m)
    Bt = workloads.random_i8((n, k), 352 + m)
    if pinned:
        A, Bt = A.pin_memory(), Bt.pin_memory()
    C = torch.full((m, n), -7, dtype=torch.int32)
    if pinned:
        C = C.pin_memory()
    plan = B.gemm_i8_plan(m, k, n)
    assert plan.path == B.GEMM_PATH_SKINNY
    ref = oracle.gemm_i8(A.numpy(), Bt.numpy())
    for _ in range(3):
        C.fill_(-7)
        B.gemm_i8_run_host(plan, A, Bt, C)
        assert np.array_equal(C.numpy(), ref)


@pytest.mark.parametrize("m,k,n,pinned", [(2048, 1024, 2048, True), (3000, 1040, 2800, False), (4096, 4096, 4096, True)])
def test_host_entry_point_banded(m, k, n, pinned):
    # at least 2048 rows and 32 MiB of copies: the band / rectangle pipeline
    A = workloads.random_i8((m, k), 27 + m)
    Bt = workloads.random_i8((n, k), 28 + n)
    C = torch.full((m, n), -7, dtype=torch.int32)
    if pinned:
        A, Bt, C = A.pin_memory(), Bt.pin_memory(), C.pin_memory()
    B.gemm_i8_run_host(B.gemm_i8_plan(m, k, n), A, Bt, C)
    G.assert_i8_exact(A, Bt, C)
    B.gemm_i8_run_host(B.gemm_i8_plan(m, k, n), A, Bt, C, torch.cuda.Stream())   # on a side stream
    G.assert_i8_exact(A, Bt, C)


@pytest.mark.parametrize("m,k,n,pinned", [
    (3000, 1040, 4500, True),    # 2 x 2 blocks, ragged bands (1500 rows; 2250 columns)
    (4100, 1000, 8300, False),   # 4 x 4 blocks, k % 16 != 0 (re-pitched f16 rows), pageable
    (2048, 4096, 4096, True),    # 2 x 2 blocks, four K chunks
    (3000, 12288, 255, True),    # narrow C (n % 4 != 0): 2 x 1 bands, rectangles split 8 ways along K
])
def test_host_entry_point_blocked_shapes(m, k, n, pinned):
    A = workloads.random_i8((m, k), 41 + m)
    Bt = workloads.random_i8((n, k), 42 + n)
    C = torch.full((m, n), -7, dtype=torch.int32)
    if pinned:
        A, Bt, C = A.pin_memory(), Bt.pin_memory(), C.pin_memory()
    B.gemm_i8_run_host(B.gemm_i8_plan(m, k, n), A, Bt, C)
    G.assert_i8_exact(A, Bt, C)


def test_host_entry_point_blocked_bf16_repitched():
    # bf16 with k % 8 != 0: each band is re-pitched once on the device
    m, k, n = 2100, 1001, 4200
    A = workloads.random_bf16((m, k), 43)
    Bt = workloads.random_bf16((n, k), 44)
    C = torch.full((m, n), float("nan"), dtype=torch.float32).pin_memory()
    B.gemm_bf16_run_host(B.gemm_bf16_plan(m, k, n), A.pin_memory(), Bt.pin_memory(), C)
    G.assert_bf16_close(A, Bt, C)


def test_host_entry_point_banded_bf16():
    m, k, n = 2304, 512, 2304
    A = workloads.random_bf16((m, k), 31)
    Bt = workloads.random_bf16((n, k), 32)
    C = torch.empty((m, n), dtype=torch.float32).pin_memory()
    B.gemm_bf16_run_host(B.gemm_bf16_plan(m, k, n), A.pin_memory(), Bt.pin_memory(), C)
    G.assert_bf16_close(A, Bt, C)


def test_misaligned_device_pointers_rejected():
    lib = B.load()
    buf = torch.zeros(4096, dtype=torch.int8, device="cuda")
    p = B.gemm_i8_plan(128, 16, 16)
    base = buf.data_ptr()
    assert lib.gemm_i8_run(ctypes.byref(p), base + 1, base, base, None) == B.GEMM_ERR_MISALIGNED
    assert lib.gemm_i8_run(ctypes.byref(p), base, base + 8, base, None) == B.GEMM_ERR_MISALIGNED


def test_trace_counts_launches():
    m, k, n = 512, 512, 512
    dA = workloads.random_i8((m, k), 27).cuda()
    dB = workloads.random_i8((n, k), 28).cuda()
    C = torch.empty((m, n), dtype=torch.int32, device="cuda")
    p = B.gemm_i8_plan(m, k, n)
    B.gemm_trace_begin(16)
    for _ in range(3):
        B.gemm_i8_run(p, dA, dB, C)
    ms, timed, cnt = B.gemm_trace_collect()
    assert cnt[B.GEMM_KERNEL_STAGE] == 3 and cnt[B.GEMM_KERNEL_TC] == 3
    assert timed == [3, 3, 0, 0] and ms[B.GEMM_KERNEL_TC] > 0
    # sampled: calls 0, 4 and 8 of 10 are timed, all launches counted
    B.gemm_trace_begin(16, 4)
    for _ in range(10):
        B.gemm_i8_run(p, dA, dB, C)
    ms, timed, cnt = B.gemm_trace_collect()
    assert cnt == [10, 10, 0, 0] and timed == [3, 3, 0, 0]
    G.assert_i8_exact(dA.cpu(), dB.cpu(), C.cpu())
    # skinny tensor-core path: staging and skinny launches timed as one unit
    ps = B.gemm_i8_plan(16, k, n)
    B.gemm_trace_begin(4)
    Cs = torch.empty((16, n), dtype=torch.int32, device="cuda")
    B.gemm_i8_run(ps, dA[:16].contiguous(), dB, Cs)
    ms, timed, cnt = B.gemm_trace_collect()
    assert cnt == [1, 0, 1, 0] and timed == [0, 0, 1, 0] and ms[B.GEMM_KERNEL_SKINNY] > 0


@pytest.mark.parametrize("bm,bn", TILES)
def test_kernel_resources_match_planner(bm, bn):
    # block_per_cu of claim 6 assumes these register counts; the compiled
    # kernels must not use more.  (The runtime's occupancy query reports one
    # CTA per SM for any kernel that allocates TMEM, although the hardware
    # co-schedules two such CTAs of this size; the planner counts registers,
    # shared memory and TMEM itself.)
    assumed = 168 if bn >= 128 else 80
    if bm == 256:
        for dtype in (B.GEMM_DTYPE_I8, B.GEMM_DTYPE_BF16):
            regs, occ = B.gemm_tc_kernel_info(bm, bn, dtype)
            assert 0 < regs <= assumed and occ >= 1
        return
    for dtype in (B.GEMM_DTYPE_I8, B.GEMM_DTYPE_BF16):
        regs, occ = B.gemm_tc_kernel_info(bm, bn, dtype)
        assert 0 < regs <= assumed
        assert occ >= 1
    p = B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, 4096, 4096, 4096, 152)
    p.bm, p.bn = bm, bn
    smem = 4 * (bm + bn) * 128 + 2048 + (8 * 4096 if (bm == 128 and bn >= 128) else 0)
    bpc = min(65536 // (384 * assumed), 233472 // smem, 512 // (2 * bn))
    # dynamic + 1 KiB reserved per CTA must fit bpc CTAs
    assert bpc * (smem + 1024) <= 233472


def test_bounded_wait_gives_up_and_reports():
    # a wait on a barrier nothing completes must end with an error status the
    # host reads, and leave the context usable
    assert B.gemm_device_error() == (B.GEMM_OK, 0)
    B.gemm_selftest_wait_timeout(20000)
    assert B.gemm_device_error() == (B.GEMM_ERR_TIMEOUT, 5)
    assert B.gemm_device_error() == (B.GEMM_OK, 0)
    A = workloads.random_i8((256, 300), 31)
    Bt = workloads.random_i8((200, 300), 32)
    G.assert_i8_exact(A, Bt, G.gpu_i8(A, Bt))


@pytest.mark.parametrize("grid,n,split", [
    (14, 1000, 3),    # 32 tiles = 2 x 14 + 4 -> 4 tiles in 3 K slices (TMA reduce-add)
    (10, 1000, 5),    # 30 + 2 -> 2 tiles in 5 slices of one chunk each
    (31, 1000, 5),    # 31 + 1 -> 1 tile in 5 slices
    (13, 998, 2),     # n % 4 != 0: direct stores and atomic adds
])
def test_i8_tail_split_exact(grid, n, split):
    # int8 tiles of the last, partial wave split along K: the staging kernel
    # zeroes C over them and every slice adds into it; bit-exact
    m, k = 1000, 4100
    A = workloads.random_i8((m, k), 41)
    Bt = workloads.random_i8((n, k), 42)
    p = forced_plan(B.GEMM_DTYPE_I8, m, k, n, 128, 256, grid)
    tiles = -(-m // 128) * -(-n // 256)
    full = tiles // grid * grid
    assert min(grid // (tiles - full), 5, 8) == split
    C1 = G.gpu_i8(A, Bt, plan=p)
    G.assert_i8_exact(A, Bt, C1)
    C2 = G.gpu_i8(A, Bt, plan=p)    # again, into a poisoned C: the zeroing happens every launch
    assert torch.equal(C1, C2)


def test_i8_tail_split_workloads_extreme():
    # 4096^3 runs 56 tail tiles in 2 K slices on 152 SMs; extreme values
    # check that the slice sums add exactly
    m = k = n = 4096
    A = torch.full((m, k), -128, dtype=torch.int8)
    Bt = torch.full((n, k), -128, dtype=torch.int8)
    Bt[::3] = 127
    C = G.gpu_i8(A, Bt)
    want = torch.full((n,), 16384 * k, dtype=torch.int32)
    want[::3] = -128 * 127 * k
    assert torch.equal(C, want.expand(m, n))


@pytest.mark.parametrize("m,k,n", [
    (1, 16, 1), (16, 64, 128), (17, 4112, 300), (33, 2048, 129), (64, 1040, 1000),
    (5, 20000, 640), (40, 8192, 8191), (64, 128, 40000),
    (65, 1024, 1000), (100, 2064, 777), (128, 8192, 4096), (127, 16, 129),
])
def test_i8_skinny_tensor_core_shapes(m, k, n):
    # k % 16 == 0: the tensor-core skinny kernel (stream-K over 128-row tiles,
    # int8 widened into TMEM, exact int32 atomics into C)
    A = workloads.random_i8((m, k), m + k)
    Bt = workloads.random_i8((n, k), n + 2 * k)
    G.assert_i8_exact(A, Bt, G.gpu_i8(A, Bt))


@pytest.mark.parametrize("m,k,n", [(1, 8192, 8192), (16, 8192, 8192), (64, 8192, 8192), (5, 3328, 2000),
                                   (128, 8192, 8192), (90, 2048, 3000)])
def test_i8_skinny_repeat_stress(m, k, n):
    # many back-to-back launches: the kernel's barrier protocol (two MMA
    # issuers and two widening groups sharing TMEM buffers and accumulators)
    # must neither time out nor mix phases under any timing
    A = workloads.random_i8((m, k), 61 + m)
    Bt = workloads.random_i8((n, k), 62 + m)
    C0 = G.gpu_i8(A, Bt)
    G.assert_i8_exact(A, Bt, C0)
    dA, dB = A.cuda(), Bt.cuda()
    p = B.gemm_i8_plan(m, k, n)
    outs = [torch.empty((m, n), dtype=torch.int32, device="cuda") for _ in range(8)]
    ref = C0.cuda()
    for it in range(400):
        B.gemm_i8_run(p, dA, dB, outs[it % 8])
        if it % 8 == 7:
            for o in outs:
                assert torch.equal(o, ref)
    assert B.gemm_device_error() == (B.GEMM_OK, 0)


def test_i8_skinny_two_streams():
    # skinny GEMMs running at the same time on two streams (each call takes
    # its own scratch from the stream-ordered pool) must not disturb each other
    shapes = [(16, 8192, 4096), (40, 4096, 8192)]
    data = []
    for i, (m, k, n) in enumerate(shapes):
        A = workloads.random_i8((m, k), 91 + i)
        Bt = workloads.random_i8((n, k), 93 + i)
        want = torch.from_numpy(oracle.gemm_i8(A.numpy(), Bt.numpy()))
        data.append((B.gemm_i8_plan(m, k, n), A.cuda(), Bt.cuda(), want,
                     [torch.empty((m, n), dtype=torch.int32, device="cuda") for _ in range(4)]))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for it in range(40):
        for (p, dA, dB, _, outs), s in zip(data, streams):
            B.gemm_i8_run(p, dA, dB, outs[it % 4], s)
    torch.cuda.synchronize()
    for (_, _, _, want, outs) in data:
        for o in outs:
            assert torch.equal(o.cpu(), want)
    assert B.gemm_device_error() == (B.GEMM_OK, 0)


@pytest.mark.parametrize("m,k,n", [
    (7, 4096, 4096),      # 32 tiles of 128 rows of Bt
    (32, 1024, 16384),    # 128 tiles, 4 stages each
    (3, 2048, 1900),      # 15 tiles, the last one ragged
    (31, 1296, 2560),     # ragged last stage (16 K)
    (17, 8192, 8192),     # m just above a 16-row MMA
])
def test_i8_skinny_more_shapes(m, k, n):
    # stream-K ranges that start and end mid-tile and mid-chunk on tiles of
    # every fill, then the extremes: every 1024-K chunk reaches 2^24
    A = workloads.random_i8((m, k), 331 + m)
    Bt = workloads.random_i8((n, k), 332 + m)
    G.assert_i8_exact(A, Bt, G.gpu_i8(A, Bt))
    A = torch.full((m, k), -128, dtype=torch.int8)
    Bt = torch.full((n, k), -128, dtype=torch.int8)
    Bt[1::3] = 127
    C = G.gpu_i8(A, Bt)
    assert torch.all(C[:, 0::3] == 16384 * k) and torch.all(C[:, 1::3] == -128 * 127 * k)


def test_i8_skinny_chain_output_feeds_next_weights():
    # Back-to-back skinny calls on one stream overlap: each call's kernels
    # start while the previous call's still run (programmatic dependent
    # launch).  Here every call's Bt is the bytes of the previous call's C,
    # so a kernel that read its Bt before the previous call had finished
    # would multiply stale bytes.  Each C is 16 x 8192 int32 = 512 KiB,
    # read as the next call's Bt of 512 x 1024 int8.
    m, k, n = 16, 8192, 8192
    m2, k2, n2 = 8, 1024, 512
    A1 = workloads.random_i8((m, k), 301)
    Bt1 = workloads.random_i8((n, k), 302)
    A2 = [workloads.random_i8((m2, k2), 303 + i) for i in range(3)]
    # the chain on the CPU: C1 = A1 Bt1; then three calls whose Bt is the
    # previous C's bytes (every one of them 512 KiB)
    C1 = oracle.gemm_i8(A1.numpy(), Bt1.numpy())
    want = [C1]
    prev = C1
    for i in range(3):
        bt = np.ascontiguousarray(prev).view(np.int8).reshape(n2, k2)
        out = oracle.gemm_i8(A2[i].numpy(), bt)
        # later links multiply a 8 x 512 C, so it is embedded in a 512 KiB
        # buffer of the previous C's remaining bytes: the GPU side does the same
        # by writing into the first rows of the buffer it reads next
        nxt = np.ascontiguousarray(prev).copy().view(np.int32).reshape(-1)
        nxt[:out.size] = out.reshape(-1)
        prev = nxt.reshape(m, n)
        want.append(out)
    bufs = [torch.full((m, n), -7, dtype=torch.int32, device="cuda") for _ in range(4)]
    dA1, dB1 = A1.cuda(), Bt1.cuda()
    dA2 = [a.cuda() for a in A2]
    p1 = B.gemm_i8_plan(m, k, n)
    p2 = B.gemm_i8_plan(m2, k2, n2)
    torch.cuda.synchronize()
    B.gemm_i8_run(p1, dA1, dB1, bufs[0])
    for i in range(3):
        # the next buffer starts as a copy of the one being read (torch's copy
        # kernel sits between the two calls), then its first rows take C
        bufs[i + 1].copy_(bufs[i])
        out = bufs[i + 1].view(-1)[: m2 * n2].view(m2, n2)
        B.gemm_i8_run(p2, dA2[i], bufs[i].view(torch.int8).view(n2, k2), out)
    torch.cuda.synchronize()
    assert np.array_equal(bufs[0].cpu().numpy(), want[0])
    for i in range(3):
        got = bufs[i + 1].view(-1)[: m2 * n2].view(m2, n2).cpu().numpy()
        assert np.array_equal(got, want[i + 1]), "link %d differs" % (i + 1)
    assert B.gemm_device_error() == (B.GEMM_OK, 0)


def test_i8_skinny_chain_direct_alias():
    # Two skinny calls back to back with nothing between them: the second
    # call's Bt is the first call's C.  Only the grid-dependency wait orders
    # the second call's reads of Bt after the first call's writes of C.
    m, k, n = 16, 8192, 8192
    m2, k2, n2 = 8, 1024, 512
    A1 = workloads.random_i8((m, k), 311)
    Bt1 = workloads.random_i8((n, k), 312)
    A2 = workloads.random_i8((m2, k2), 313)
    C1 = oracle.gemm_i8(A1.numpy(), Bt1.numpy())
    want2 = oracle.gemm_i8(A2.numpy(), np.ascontiguousarray(C1).view(np.int8).reshape(n2, k2))
    dA1, dB1, dA2 = A1.cuda(), Bt1.cuda(), A2.cuda()
    p1 = B.gemm_i8_plan(m, k, n)
    p2 = B.gemm_i8_plan(m2, k2, n2)
    for rep in range(20):
        C = torch.full((m, n), -7, dtype=torch.int32, device="cuda")
        C2 = torch.full((m2, n2), -7, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        B.gemm_i8_run(p1, dA1, dB1, C)
        B.gemm_i8_run(p2, dA2, C.view(torch.int8).view(n2, k2), C2)
        torch.cuda.synchronize()
        assert np.array_equal(C.cpu().numpy(), C1)
        assert np.array_equal(C2.cpu().numpy(), want2), "repetition %d" % rep
    assert B.gemm_device_error() == (B.GEMM_OK, 0)


def test_i8_mixed_paths_chain_direct_alias():
    # tensor path -> skinny path -> tensor path, back to back on one stream,
    # each call reading the previous call's C (its bytes) as an operand:
    #   C1 = A1 Bt1        (256 x 512, tensor path)      512 KiB
    #   C2 = A2 (C1 as Bt) (8 x 512, skinny path)        16 KiB, Bt = 512 x 1024
    #   C3 = (C2 as A) Bt3 (256 x 96, tensor path)       A = 256 x 64
    A1 = workloads.random_i8((256, 512), 341)
    Bt1 = workloads.random_i8((512, 512), 342)
    A2 = workloads.random_i8((8, 1024), 343)
    Bt3 = workloads.random_i8((96, 64), 344)
    C1 = oracle.gemm_i8(A1.numpy(), Bt1.numpy())
    C2 = oracle.gemm_i8(A2.numpy(), np.ascontiguousarray(C1).view(np.int8).reshape(512, 1024))
    C3 = oracle.gemm_i8(np.ascontiguousarray(C2).view(np.int8).reshape(256, 64), Bt3.numpy())
    p1, p2, p3 = B.gemm_i8_plan(256, 512, 512), B.gemm_i8_plan(8, 1024, 512), B.gemm_i8_plan(256, 64, 96)
    assert (p1.path, p2.path, p3.path) == (B.GEMM_PATH_TENSOR, B.GEMM_PATH_SKINNY, B.GEMM_PATH_TENSOR)
    dA1, dB1, dA2, dB3 = A1.cuda(), Bt1.cuda(), A2.cuda(), Bt3.cuda()
    for rep in range(10):
        g1 = torch.full((256, 512), -7, dtype=torch.int32, device="cuda")
        g2 = torch.full((8, 512), -7, dtype=torch.int32, device="cuda")
        g3 = torch.full((256, 96), -7, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        B.gemm_i8_run(p1, dA1, dB1, g1)
        B.gemm_i8_run(p2, dA2, g1.view(torch.int8).view(512, 1024), g2)
        B.gemm_i8_run(p3, g2.view(torch.int8).view(256, 64), dB3, g3)
        torch.cuda.synchronize()
        assert np.array_equal(g1.cpu().numpy(), C1)
        assert np.array_equal(g2.cpu().numpy(), C2), "skinny link, repetition %d" % rep
        assert np.array_equal(g3.cpu().numpy(), C3), "tensor link, repetition %d" % rep
    assert B.gemm_device_error() == (B.GEMM_OK, 0)


@pytest.mark.parametrize("m,k,n", [(16, 4096, 1024), (100, 2048, 640)])
def test_i8_skinny_c_offset(m, k, n):
    # C starting 4 bytes into an allocation (C needs only 4-byte alignment):
    # every element written exactly, nothing outside C touched
    A = workloads.random_i8((m, k), 321 + m)
    Bt = workloads.random_i8((n, k), 322 + m)
    base = torch.full((m * n + 4,), -7, dtype=torch.int32, device="cuda")
    C = base[1:1 + m * n].view(m, n)
    B.gemm_i8_run(B.gemm_i8_plan(m, k, n), A.cuda(), Bt.cuda(), C)
    torch.cuda.synchronize()
    G.assert_i8_exact(A, Bt, C.cpu())
    assert base[0].item() == -7 and torch.all(base[1 + m * n:] == -7)


@pytest.mark.parametrize("m", [64, 128])
def test_i8_skinny_extremes(m):
    k, n = 16384, 1000
    A = torch.full((m, k), -128, dtype=torch.int8)
    Bt = torch.full((n, k), -128, dtype=torch.int8)
    Bt[1::2] = 127
    C = G.gpu_i8(A, Bt)
    assert torch.all(C[:, 0::2] == 16384 * k)
    assert torch.all(C[:, 1::2] == -128 * 127 * k)


@pytest.mark.parametrize("m,k,n,grid", [
    (4096, 4096, 4096, 152), (1000, 3000, 777, 20), (513, 2100, 1500, 6), (257, 64, 300, 2),
])
def test_i8_two_sm_tile_shapes(m, k, n, grid):
    # the 256 x 256 two-SM tile on ragged shapes and persistent grids
    A = workloads.random_i8((m, k), m + 17)
    Bt = workloads.random_i8((n, k), n + 19)
    p = forced_plan(B.GEMM_DTYPE_I8, m, k, n, 256, 256, grid)
    G.assert_i8_exact(A, Bt, G.gpu_i8(A, Bt, plan=p))


@pytest.mark.parametrize("k,n,grid,split", [
    (4100, 1500, 14, 2),    # 24 tiles = 3 x 7 pairs + 3 -> 3 tiles in 2 K slices
    (4100, 1500, 22, 5),    # 2 x 11 + 2 -> 2 tiles in 5 slices (the last one a single K step)
    (4100, 1500, 46, 5),    # 23 + 1, capped by the 5 K chunks
    (8200, 1500, 46, 8),    # 9 K chunks: capped at 8 slices
    (4100, 1498, 14, 2),    # n % 4 != 0: direct stores of C
])
def test_i8_two_sm_tail_split_exact(k, n, grid, split):
    # two-SM tiles of the last, partial round split along K over idle pairs:
    # every slice adds into C, zeroed over those tiles by the staging kernel
    m = 1000
    A = workloads.random_i8((m, k), 51)
    Bt = workloads.random_i8((n, k), 52)
    p = forced_plan(B.GEMM_DTYPE_I8, m, k, n, 256, 256, grid)
    tiles = -(-m // 256) * -(-n // 256)
    pairs = grid // 2
    nch = -(-(-(-k // 64)) // 16)
    assert min(pairs // (tiles - tiles // pairs * pairs), nch, 8) == split
    C1 = G.gpu_i8(A, Bt, plan=p)
    G.assert_i8_exact(A, Bt, C1)
    C2 = G.gpu_i8(A, Bt, plan=p)    # again, into a poisoned C
    assert torch.equal(C1, C2)
    assert B.gemm_device_error() == (B.GEMM_OK, 0)


@pytest.mark.parametrize("m,k,n", [(1000, 3000, 777), (512, 1024, 516)])
def test_bf16_two_sm_tile_shapes(m, k, n):
    A = workloads.random_bf16((m, k), m + 23)
    Bt = workloads.random_bf16((n, k), n + 29)
    p = forced_plan(B.GEMM_DTYPE_BF16, m, k, n, 256, 256, 8)
    G.assert_bf16_close(A, Bt, G.gpu_bf16(A, Bt, plan=p))


# Two-SM (256 x 256) int8 tiles with k % 16 == 0: ragged m, n and k (a last
# K chunk of 16 elements), persistent grids with many tiles per pair, a
# single tile, and C that TMA cannot store (n % 4 != 0).
@pytest.mark.parametrize("m,k,n,grid", [
    (1000, 2064, 1000, 8),     # 4 x 4 tiles on 4 pairs; K = 1024 + 1024 + 16
    (513, 1040, 4100, 6),      # 3 x 17 tiles on 3 pairs; last tile column 4 wide
    (300, 128, 230, 2),        # two K steps; one tile column, 230 wide
    (1024, 4096, 1002, 152),   # n % 4 != 0: direct stores of C
    (256, 8192, 224, 2),       # exactly one tile, eight K chunks
    (2048, 1024, 2560, 152),   # 80 tiles on 76 pairs; one K chunk, so no tail split
])
def test_i8_two_sm_k16_shapes(m, k, n, grid):
    A = workloads.random_i8((m, k), m + 29)
    Bt = workloads.random_i8((n, k), n + 31)
    p = forced_plan(B.GEMM_DTYPE_I8, m, k, n, 256, 256, grid)
    C1 = G.gpu_i8(A, Bt, plan=p)
    G.assert_i8_exact(A, Bt, C1)
    C2 = G.gpu_i8(A, Bt, plan=p)
    assert torch.equal(C1, C2)
    assert B.gemm_device_error() == (B.GEMM_OK, 0)


@pytest.mark.parametrize("a,b", [(-128, -128), (-128, 127), (127, 127)])
def test_i8_two_sm_chunk_extremes(a, b):
    # on the two-SM tile, every 1024-element chunk sums to +-2^24 (or just
    # below): exact only if each chunk is drained before fp32 would round
    m, k, n = 512, 8192, 448
    A = torch.full((m, k), a, dtype=torch.int8)
    Bt = torch.full((n, k), b, dtype=torch.int8)
    p = forced_plan(B.GEMM_DTYPE_I8, m, k, n, 256, 256, 4)
    C = G.gpu_i8(A, Bt, plan=p)
    assert torch.all(C == a * b * k)
    Bt[1::2] = -b if b != -128 else 127
    C = G.gpu_i8(A, Bt, plan=p)
    assert torch.all(C[:, 0::2] == a * b * k)
    assert torch.all(C[:, 1::2] == a * int(Bt[1, 0]) * k)


# Small-MN, large-K int8 problems: the planner splits every two-SM tile along
# K and every slice adds into C zeroed by the staging kernel.
@pytest.mark.parametrize("m,k,n", [
    (512, 8192, 512),      # 4 tiles x 8 slices
    (1000, 4096, 300),     # 8 tiles x 4 slices; n % 4 != 0: slices add with atomics
    (200, 4096, 4096),     # 16 tiles x 4 slices, one ragged tile row
    (700, 3000, 900),      # k % 16 != 0 (re-pitched rows); 12 tiles x 2 slices of 23-24 K steps
])
def test_i8_k_split_plans_exact(m, k, n):
    p = B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, m, k, n, torch.cuda.get_device_properties(0).multi_processor_count)
    assert p.bm == 256 and p.split_k >= 2 and p.split_from == 0
    A = workloads.random_i8((m, k), m + 61)
    Bt = workloads.random_i8((n, k), n + 62)
    C1 = G.gpu_i8(A, Bt, plan=p)
    G.assert_i8_exact(A, Bt, C1)
    C2 = G.gpu_i8(A, Bt, plan=p)   # again, into a poisoned C
    assert torch.equal(C1, C2)
    assert B.gemm_device_error() == (B.GEMM_OK, 0)


def test_i8_k_split_extremes_exact():
    # 8 slices of 8192 K elements each, every chunk at +2^24: C = 2^30
    m, k, n = 300, 65536, 300
    p = B.gemm_plan_for_sms(B.GEMM_DTYPE_I8, m, k, n, torch.cuda.get_device_properties(0).multi_processor_count)
    assert p.split_k == 8 and p.split_from == 0
    A = torch.full((m, k), -128, dtype=torch.int8)
    Bt = torch.full((n, k), -128, dtype=torch.int8)
    C = G.gpu_i8(A, Bt, plan=p)
    assert torch.all(C == 16384 * k)


@pytest.mark.parametrize("bm,bn", [(128, 128), (128, 256), (256, 256)])
@pytest.mark.parametrize("grid", [6, 1000])
def test_wide_tiles_unaligned_c(bm, bn, grid):
    # n % 4 != 0: C cannot take TMA stores; the wide tiles transpose each
    # 32 x 32 block through shared memory into stores / atomics along rows
    # (grid 6: tail split, slices add; grid 1000: plain stores, then every
    # tile split 2 ways)
    m, k, n = 900, 2100, 701
    A = workloads.random_i8((m, k), 71)
    Bt = workloads.random_i8((n, k), 72)
    if grid == 1000:
        ps = forced_plan(B.GEMM_DTYPE_I8, m, k, n, bm, bn, grid, 2)
        G.assert_i8_exact(A, Bt, G.gpu_i8(A, Bt, plan=ps))
    p = forced_plan(B.GEMM_DTYPE_I8, m, k, n, bm, bn, grid)
    C1 = G.gpu_i8(A, Bt, plan=p)
    G.assert_i8_exact(A, Bt, C1)
    assert torch.equal(C1, G.gpu_i8(A, Bt, plan=p))
    Ab = workloads.random_bf16((m, 1000), 73)
    Bb = workloads.random_bf16((n, 1000), 74)
    pb = forced_plan(B.GEMM_DTYPE_BF16, m, 1000, n, bm, bn, grid)
    G.assert_bf16_close(Ab, Bb, G.gpu_bf16(Ab, Bb, plan=pb))


# ----------------------------------------------- int8 A widened on chip ----

def a_on_chip_plan(m, k, n, on=1, split=None, grid=None):
    # the planner's plan with A widened inside the two-SM kernel (or not)
    p = B.gemm_i8_plan(m, k, n)
    p.bm, p.bn = 256, 256
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    tiles = -(-m // 256) * -(-n // 256)
    p.grid = 2 * min(tiles, pairs) if grid is None else grid
    if split is not None:
        if split > 1:
            p.split_k, p.split_from = split, 0
        else:
            p.split_k, p.split_from = 1, max(1, tiles)
    p.a_on_chip = on
    return p


@pytest.mark.parametrize("m,k,n,split", [
    (4097, 16384, 255, None),   # the planned narrow shape (every tile split 4 ways along K)
    (300, 2096, 700, 1),        # ragged rows and columns, k % 64 = 48
    (513, 1024, 257, 3),        # K slices of 5-6 steps, ragged tile edges
    (1000, 4096, 512, 1),
    (2048, 8192, 128, 4),
    (256, 16, 256, 1),          # a single K step of 16
    (640, 3072, 1000, None),    # planned tile with a tail split
])
def test_i8_a_on_chip(m, k, n, split):
    A = workloads.random_i8((m, k), 201)
    Bt = workloads.random_i8((n, k), 202)
    p = a_on_chip_plan(m, k, n, 1, split)
    G.assert_i8_exact(A, Bt, G.gpu_i8(A, Bt, plan=p))


@pytest.mark.parametrize("m,k,n,split,grid", [
    (2000, 1936, 500, 1, 4),    # 16 whole tiles of 31 K steps (odd) on 2 pairs
    (700, 3008, 300, 3, 2),     # 6 tiles x 3 K slices of 15-16 steps on one pair
    (2000, 1936, 255, 1, 4),    # odd n <= 256 but more units than pairs: the
    (700, 3008, 255, 3, 2),     # rings with C staging, runs only for the last unit
])
def test_i8_a_on_chip_many_units_per_pair(m, k, n, split, grid):
    # each pair runs several units back to back, so the int8 boxes of one
    # unit follow another's in the same ring, also after an odd step count
    A = workloads.random_i8((m, k), 204)
    Bt = workloads.random_i8((n, k), 205)
    p = a_on_chip_plan(m, k, n, 1, split, grid)
    G.assert_i8_exact(A, Bt, G.gpu_i8(A, Bt, plan=p))


@pytest.mark.parametrize("on", [0, 1])
@pytest.mark.parametrize("n,offset,split", [(255, 1, 3), (256, 1, 3), (257, 3, 3), (255, 2, 3), (384, 3, 3),
                                            (255, 0, 1), (200, 1, 1), (129, 2, 1), (300, 3, 1), (1, 0, 3)])
def test_i8_pair_unaligned_c(n, offset, split, on):
    # the two-SM kernel writing (whole tiles) or adding (K-split tiles) into a
    # C whose rows are not 16-byte aligned (n % 4 != 0, or C starting 4-12
    # bytes into its allocation): with odd n <= 256 a CTA's rows go out as
    # one contiguous run by bulk copies or reduce-adds, other split tiles row
    # by row; the unaligned ends by plain stores or atomics; every element
    # exact, nothing outside C touched
    m, k = 513, 2048
    A = workloads.random_i8((m, k), 206 + n)
    Bt = workloads.random_i8((n, k), 207 + offset)
    p = a_on_chip_plan(m, k, n, on, split)
    base = torch.full((m * n + 8,), -7, dtype=torch.int32, device="cuda")
    C = base[offset:offset + m * n].view(m, n)
    B.gemm_i8_run(p, A.cuda(), Bt.cuda(), C)
    torch.cuda.synchronize()
    G.assert_i8_exact(A, Bt, C.cpu())
    assert torch.all(base[:offset] == -7) and torch.all(base[offset + m * n:] == -7)
    assert B.gemm_device_error() == (B.GEMM_OK, 0)


def test_i8_a_on_chip_extremes_and_repeat():
    # all -128 (every fp32 chunk reaches exactly 2^24) and alternating signs,
    # twice in a row into a poisoned C
    m, k, n = 512, 16384, 256
    A = torch.full((m, k), -128, dtype=torch.int8)
    Bt = torch.full((n, k), -128, dtype=torch.int8)
    p = a_on_chip_plan(m, k, n, 1)
    C = G.gpu_i8(A, Bt, plan=p)
    assert bool((C == 16384 * k).all())
    A2 = workloads.random_i8((m, k), 203)
    Bt2 = (torch.arange(n * k, dtype=torch.int64).reshape(n, k) % 2 * 254 - 127).to(torch.int8)
    for _ in range(2):
        G.assert_i8_exact(A2, Bt2, G.gpu_i8(A2, Bt2, plan=p))


def test_i8_a_on_chip_planned_and_rejected():
    # the planner widens A on chip for narrow C on the two-SM tile only, and
    # gemm_i8_run refuses the flag where the kernel cannot widen
    assert B.gemm_i8_plan(4097, 16384, 255).a_on_chip == 1
    assert B.gemm_i8_plan(8192, 8192, 8192).a_on_chip == 0
    import ctypes
    lib = B.load()
    buf = torch.zeros(1 << 20, dtype=torch.int8, device="cuda")
    for m, k, n in [(4097, 16384, 255), (1000, 777, 3000)]:
        p = B.gemm_i8_plan(m, k, n)
        p.a_on_chip = 1
        if p.bm == 256 and k % 16 == 0:
            p.bm, p.bn = 128, 128
        st = lib.gemm_i8_run(ctypes.byref(p), buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), None)
        assert st == B.GEMM_ERR_INVALID_ARG
