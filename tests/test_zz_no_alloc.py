"""The allocation-free int8 entry point, gemm_i8_run_noalloc, against
gemm_i8_run.

Some callers cannot let a library allocate device memory (memory-planned
runtimes, latency-critical loops); for them gemm_i8_run_noalloc stages its
f16 operand copies in a fixed static device array instead of a memory pool.
Its results must equal gemm_i8_run's bit for bit, on consecutive calls that
reuse the shared array.  This file is collected last on purpose."""

import ctypes

import pytest
import torch

from dense_int8_matrix_gb300 import binding as B
from dense_int8_matrix_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_int8_matrix_gb300 import build
    build.build()
    B.load()


def _both(m, k, n, seed):
    A = workloads.random_i8((m, k), seed).cuda()
    Bt = workloads.random_i8((n, k), seed + 1).cuda()
    plan = B.gemm_i8_plan(m, k, n)
    ref = torch.empty((m, n), dtype=torch.int32, device="cuda")
    B.gemm_i8_run(plan, A, Bt, ref)
    out = torch.full((m, n), -7, dtype=torch.int32, device="cuda")
    lib = B.load()
    st = lib.gemm_i8_run_noalloc(ctypes.byref(plan), A.data_ptr(), Bt.data_ptr(), out.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    assert st == B.GEMM_OK, B.gemm_status_string(st)
    torch.cuda.synchronize()
    return out, ref


def test_noalloc_matches_allocating_entry_point_twice():
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
