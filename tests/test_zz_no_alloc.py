"""The allocation-free int8 entry point, gemm_i8_run_noalloc.

Some callers cannot let a library allocate device memory: runtimes that plan
every byte of device memory up front, and latency-critical loops where an
allocation could block or fail.  For them gemm_i8_run_noalloc stages its f16
operand copies in a fixed static device array instead of a memory pool.

Checked here: results bit-exact against the CPU oracle and equal to
gemm_i8_run's, on consecutive calls that reuse the shared array; no use of
the library's pool during a call; a time-out recorded before a call stays
readable through gemm_device_error.  This file is collected last on purpose."""

import ctypes

import pytest
import torch

import oracle
from dense_int8_matrix_gb300 import binding as B
from dense_int8_matrix_gb300 import workloads
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_int8_matrix_gb300 import build
    build.build()
    oracle.build()
    B.load()
    yield
    st, code = B.gemm_device_error()
    assert st == B.GEMM_OK, "device error word set: code %d" % code


def _noalloc(plan, A, Bt):
    m, n = plan.m, plan.n
    out = torch.full((m, n), -7, dtype=torch.int32, device="cuda")   # poison
    lib = B.load()
    st = lib.gemm_i8_run_noalloc(ctypes.byref(plan), A.data_ptr(), Bt.data_ptr(), out.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    assert st == B.GEMM_OK, B.gemm_status_string(st)
    torch.cuda.synchronize()
    return out


def _both(m, k, n, seed, against_oracle=True):
    hA = workloads.random_i8((m, k), seed)
    hB = workloads.random_i8((n, k), seed + 1)
    A, Bt = hA.cuda(), hB.cuda()
    plan = B.gemm_i8_plan(m, k, n)
    ref = torch.empty((m, n), dtype=torch.int32, device="cuda")
    B.gemm_i8_run(plan, A, Bt, ref)
    out = _noalloc(plan, A, Bt)
    if against_oracle:
        G.assert_i8_exact(hA, hB, out.cpu())
    return out, ref


def test_noalloc_matches_oracle_and_allocating_entry_point_twice():
    # two calls in a row through the C ABI; the second reuses the static
    # scratch the first one filled (different shapes, so stale contents
    # would show)
    for m, k, n, seed in [(1000, 2100, 3000, 11), (700, 777, 520, 12)]:
        out, ref = _both(m, k, n, seed)
        assert torch.equal(out, ref)


def test_noalloc_largest_problem_and_rejection():
    # 4096^3 needs exactly the 64 MiB of scratch
    out, ref = _both(4096, 4096, 4096, 13)
    assert torch.equal(out, ref)
    lib = B.load()
    plan = B.gemm_i8_plan(4096, 4104, 4096)        # needs more than 64 MiB
    buf = torch.empty(16, dtype=torch.int8, device="cuda")
    st = lib.gemm_i8_run_noalloc(ctypes.byref(plan), buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), None)
    assert st == B.GEMM_ERR_INVALID_ARG


def test_noalloc_rejects_what_gemm_i8_run_rejects():
    # the same plan checks as gemm_i8_run: an out-of-range K split and an
    # empty skinny grid are refused, and nothing is launched
    lib = B.load()
    buf = torch.zeros(1 << 20, dtype=torch.int8, device="cuda")
    plan = B.gemm_i8_plan(512, 1024, 512)
    plan.split_k = 9
    st = lib.gemm_i8_run_noalloc(ctypes.byref(plan), buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), None)
    assert st == B.GEMM_ERR_INVALID_ARG
    plan = B.gemm_i8_plan(16, 1024, 256)
    assert plan.path == B.GEMM_PATH_SKINNY
    plan.grid = 0
    st = lib.gemm_i8_run_noalloc(ctypes.byref(plan), buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), None)
    assert st == B.GEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("m,k,n", [(16, 4096, 1000), (100, 4096, 1000), (64, 8192, 8192), (8, 1000, 777)])
def test_noalloc_skinny_plan(m, k, n):
    # skinny plans: the tensor-core kernel with the f16 copy of A in the static
    # array (k % 16 == 0), else the CUDA-core kernel, which needs no scratch
    out, ref = _both(m, k, n, 14 + m)
    assert torch.equal(out, ref)


def test_noalloc_skinny_twice_then_tensor():
    # consecutive calls of both paths through the shared array: stale
    # contents from the call before would show
    for m, k, n, seed in [(32, 2048, 3000, 41), (5, 4096, 640, 42), (300, 1024, 500, 43), (16, 1024, 2000, 44)]:
        out, ref = _both(m, k, n, seed)
        assert torch.equal(out, ref)


@pytest.mark.parametrize("m,k,n", [(512, 8192, 512), (1000, 4096, 300)])
def test_noalloc_k_split_plan(m, k, n):
    # small-MN, large-K plans split every two-SM tile along K; the staging
    # kernel zeroes C in the allocation-free variant too
    assert B.gemm_i8_plan(m, k, n).split_k >= 2
    out, ref = _both(m, k, n, 20 + m)
    assert torch.equal(out, ref)


def test_noalloc_plan_that_widens_a_on_chip():
    # a plan with a_on_chip = 1 runs on the staged path here (the f16 copy of
    # A in the static array), with the same result
    plan = B.gemm_i8_plan(2048, 4096, 255)
    assert plan.a_on_chip == 1
    out, ref = _both(2048, 4096, 255, 90)
    assert torch.equal(out, ref)


def test_noalloc_takes_nothing_from_the_pool():
    # the library pool's high-water mark stays at zero across tensor-path and
    # skinny calls of the allocation-free entry point, while one gemm_i8_run
    # of the same problem raises it (so the probe can see an allocation)
    shapes = [(1000, 2048, 3000), (64, 4096, 2048)]
    inputs = []
    for i, (m, k, n) in enumerate(shapes):
        inputs.append((B.gemm_i8_plan(m, k, n), workloads.random_i8((m, k), 60 + i).cuda(),
                       workloads.random_i8((n, k), 70 + i).cuda()))
    for plan, A, Bt in inputs:
        _noalloc(plan, A, Bt)      # first call per device: symbol look-up
    torch.cuda.synchronize()
    B.gemm_pool_usage(reset_high=True)
    _, high = B.gemm_pool_usage()
    assert high == 0
    for plan, A, Bt in inputs:
        _noalloc(plan, A, Bt)
    torch.cuda.synchronize()
    _, high = B.gemm_pool_usage()
    assert high == 0, "gemm_i8_run_noalloc used %d bytes of the pool" % high
    plan, A, Bt = inputs[0]
    C = torch.empty((plan.m, plan.n), dtype=torch.int32, device="cuda")
    B.gemm_i8_run(plan, A, Bt, C)
    torch.cuda.synchronize()
    _, high = B.gemm_pool_usage(reset_high=True)
    assert high >= plan.workspace_bytes > 0


def test_noalloc_keeps_a_recorded_time_out_readable():
    # the allocation-free entry point writes time-outs into the device error
    # word every entry point shares; a call neither hides nor clears a code
    # recorded before it: the self-test's bounded wait gives up (code 5),
    # then an allocation-free call runs, and gemm_device_error still reports
    B.gemm_selftest_wait_timeout(20000)
    out, ref = _both(300, 1024, 500, 80, against_oracle=False)
    assert torch.equal(out, ref)
    st, code = B.gemm_device_error()
    assert st == B.GEMM_ERR_TIMEOUT and code == 5
    st, code = B.gemm_device_error()
    assert st == B.GEMM_OK and code == 0
