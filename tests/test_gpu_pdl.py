"""Launch chaining against a producer that lets its dependents start early.

The library's kernels are launched with programmatic stream serialization, so
they may start before the kernel in front of them ends.  A producer that
triggers its dependents at once and writes a GEMM's operand only ~50 us later
(tests/cuda/late_writer.cu) must still be seen: every kernel of a call reads
its operands only after its grid dependency wait.  Skinny calls (prologue +
skinny kernel) and tensor-path calls, with the late write to Bt or to A.

What this can catch, measured on GB300 with copies of the library that had a
wait removed: the skinny prologue and the tensor path's staging kernel start
while the producer still waits, and without their own wait they read the old
operand (the skinny A case and both tensor-path cases fail).  The skinny
kernel behind the prologue did not start before the producer had ended, so
the skinny Bt cases pin the result but would not catch a missing wait in the
skinny kernel itself."""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from dense_int8_matrix_gb300 import binding as B
from dense_int8_matrix_gb300 import workloads

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def writer():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_int8_matrix_gb300 import build
    build.build()
    oracle.build()
    B.load()
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "liblate_writer.so")
    src = os.path.join(HERE, "cuda", "late_writer.cu")
    if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        subprocess.run([build.nvcc_path(), "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared",
                        "-Xcompiler", "-fPIC", "-o", so, src], check=True)
    lib = ctypes.CDLL(so)
    lib.late_writer.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p]
    lib.late_writer.restype = ctypes.c_int
    yield lib
    assert B.gemm_device_error() == (B.GEMM_OK, 0)


@pytest.mark.parametrize("m,k,n,target", [
    (8, 8192, 8192, "Bt"),      # skinny: prologue + skinny kernel
    (8, 8192, 8192, "A"),
    (64, 4096, 4096, "Bt"),
    (1000, 2048, 1500, "Bt"),   # tensor path: staging + GEMM
    (1000, 2048, 1500, "A"),
])
def test_late_operand_write_is_seen(writer, m, k, n, target):
    A_old = workloads.random_i8((m, k), 361)
    A_new = workloads.random_i8((m, k), 362)
    Bt_old = workloads.random_i8((n, k), 363)
    Bt_new = workloads.random_i8((n, k), 364)
    want = oracle.gemm_i8((A_new if target == "A" else A_old).numpy(),
                          (Bt_new if target == "Bt" else Bt_old).numpy())
    plan = B.gemm_i8_plan(m, k, n)
    stream = torch.cuda.current_stream()
    for rep in range(5):
        dA, dB = A_old.cuda(), Bt_old.cuda()
        src = (A_new if target == "A" else Bt_new).cuda()
        dst = dA if target == "A" else dB
        C = torch.full((m, n), -7, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        assert writer.late_writer(dst.data_ptr(), src.data_ptr(), dst.numel(), 50_000, stream.cuda_stream) == 0
        B.gemm_i8_run(plan, dA, dB, C, stream)
        torch.cuda.synchronize()
        assert np.array_equal(C.cpu().numpy(), want), "repetition %d" % rep
