"""Helpers shared by the GPU parity tests: run the CUDA path through the C
ABI and compare with the oracle."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from dense_int8_matrix_gb300 import binding as B


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def gpu_i8(A: torch.Tensor, Bt: torch.Tensor, plan=None, stream=None) -> torch.Tensor:
    m, k = A.shape
    n = Bt.shape[0]
    if plan is None:
        plan = B.gemm_i8_plan(m, k, n)
    dA, dB = A.cuda(), Bt.cuda()
    C = torch.full((m, n), -7, dtype=torch.int32, device="cuda")   # poison: every element must be written
    B.gemm_i8_run(plan, dA, dB, C, stream)
    torch.cuda.synchronize()
    return C.cpu()


def gpu_bf16(A: torch.Tensor, Bt: torch.Tensor, plan=None, stream=None) -> torch.Tensor:
    m, k = A.shape
    n = Bt.shape[0]
    if plan is None:
        plan = B.gemm_bf16_plan(m, k, n)
    dA, dB = A.cuda(), Bt.cuda()
    C = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    B.gemm_bf16_run(plan, dA, dB, C, stream)
    torch.cuda.synchronize()
    return C.cpu()


def assert_i8_exact(A: torch.Tensor, Bt: torch.Tensor, C: torch.Tensor):
    ref = oracle.gemm_i8(A.numpy(), Bt.numpy())
    got = C.numpy()
    if not np.array_equal(got, ref):
        bad = np.argwhere(got != ref)
        i, j = bad[0]
        raise AssertionError("%d of %d elements differ; first at (%d, %d): gpu %d oracle %d"
                             % (len(bad), got.size, i, j, got[i, j], ref[i, j]))


def assert_bf16_close(A: torch.Tensor, Bt: torch.Tensor, C: torch.Tensor, tol: float = 1e-3):
    ref, S = oracle.gemm_bf16(bits(A), bits(Bt))
    got = C.numpy().astype(np.float64)
    err = np.abs(got - ref.astype(np.float64))
    bound = tol * S
    ok = err <= bound
    if not np.all(ok):
        bad = np.argwhere(~ok)
        i, j = bad[0]
        raise AssertionError("%d elements outside |err| <= %g*S; first (%d,%d): gpu %r oracle %r S %r"
                             % (len(bad), tol, i, j, got[i, j], ref[i, j], S[i, j]))


def sample_positions(m: int, n: int, count: int, seed: int):
    rng = np.random.default_rng(seed)
    rows = rng.integers(0, m, size=count)
    cols = rng.integers(0, n, size=count)
    # always include the four corners and the last row / column
    rows = np.concatenate([rows, [0, 0, m - 1, m - 1]])
    cols = np.concatenate([cols, [0, n - 1, 0, n - 1]])
    return rows.astype(np.int64), cols.astype(np.int64)


def freivalds_i8(A: torch.Tensor, Bt: torch.Tensor, C: torch.Tensor, trials: int = 3, seed: int = 0):
    """C r == A (B r) for random r with entries in [-1024, 1024].  Every sum
    stays below 2^53 for k <= 16384 and n <= 16384, so float64 BLAS is exact."""
    rng = np.random.default_rng(seed)
    A64 = A.numpy().astype(np.float64)
    B64 = Bt.numpy().astype(np.float64)
    C64 = C.numpy().astype(np.float64)
    for _ in range(trials):
        r = rng.integers(-1024, 1025, size=C64.shape[1]).astype(np.float64)
        lhs = C64 @ r
        rhs = A64 @ (B64.T @ r)
        assert np.array_equal(lhs, rhs), "Freivalds check failed"
