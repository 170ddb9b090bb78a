"""CPU oracle for the dense GEMM (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library: the arithmetic lives in ``oracle_gemm.c`` (plain C, compiled here
with gcc) and the tile-selector reading in ``selector.py``.

The numpy wrappers below only marshal arguments.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_gemm.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

OK = 0
ERR_ARG = 1
ERR_OVERFLOW = 2


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile oracle_gemm.c into liboracle.so (gcc, portable flags only)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    # -ffp-contract=off: every float operation is rounded on its own
    cmd = ["gcc", "-O3", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_gemm_i8.argtypes = [i64, i64, i64, p, p, p, ctypes.c_int]
    lib.oracle_gemm_bf16.argtypes = [i64, i64, i64, p, p, p, p, ctypes.c_int]
    lib.oracle_gemm_i8_entries.argtypes = [i64, i64, i64, p, p, i64, p, p, p]
    lib.oracle_gemm_bf16_entries.argtypes = [i64, i64, i64, p, p, i64, p, p, p, p]
    lib.oracle_requant.argtypes = [i64, i64, p, p, p, ctypes.c_int, p]
    for f in (lib.oracle_gemm_i8, lib.oracle_gemm_bf16,
              lib.oracle_gemm_i8_entries, lib.oracle_gemm_bf16_entries, lib.oracle_requant):
        f.restype = ctypes.c_int
    _lib = lib
    return lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a.size else None


def _check(rc: int):
    if rc == ERR_OVERFLOW:
        raise OracleError("exact sum outside int32")
    if rc != OK:
        raise OracleError("oracle status %d" % rc)


def _as(a, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError("expected %s, got %s" % (dtype, a.dtype))
    return a


def gemm_i8(A, Bt, nthreads: int | None = None) -> np.ndarray:
    """C = A x B for A (m x k int8) and Bt (n x k int8, B stored K-major).
    Exact int64 sums, checked to fit int32."""
    A = _as(A, np.int8)
    Bt = _as(Bt, np.int8)
    m, k = A.shape
    n, k2 = Bt.shape
    if k != k2:
        raise ValueError("k mismatch")
    C = np.empty((m, n), dtype=np.int32)
    rc = _load().oracle_gemm_i8(m, k, n, _ptr(A), _ptr(Bt), _ptr(C),
                                nthreads or default_threads())
    _check(rc)
    return C


def gemm_bf16(A_bits, Bt_bits, nthreads: int | None = None, with_abs: bool = True):
    """C = A x B for bf16 inputs given as uint16 bit patterns.
    Returns (C float32, S float64 = sum |a*b|) or C alone."""
    A = _as(A_bits, np.uint16)
    Bt = _as(Bt_bits, np.uint16)
    m, k = A.shape
    n, k2 = Bt.shape
    if k != k2:
        raise ValueError("k mismatch")
    C = np.empty((m, n), dtype=np.float32)
    S = np.empty((m, n), dtype=np.float64) if with_abs else None
    rc = _load().oracle_gemm_bf16(m, k, n, _ptr(A), _ptr(Bt), _ptr(C),
                                  _ptr(S) if S is not None else None,
                                  nthreads or default_threads())
    _check(rc)
    return (C, S) if with_abs else C


def gemm_i8_entries(A, Bt, rows, cols) -> np.ndarray:
    """Exact int64 C[rows[t], cols[t]] for sampled positions."""
    A = _as(A, np.int8)
    Bt = _as(Bt, np.int8)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    out = np.empty(rows.shape[0], dtype=np.int64)
    m, k = A.shape
    n = Bt.shape[0]
    rc = _load().oracle_gemm_i8_entries(m, k, n, _ptr(A), _ptr(Bt), rows.shape[0],
                                        _ptr(rows), _ptr(cols), _ptr(out))
    _check(rc)
    return out


def gemm_bf16_entries(A_bits, Bt_bits, rows, cols):
    """(double sum, double sum |a*b|) at sampled positions."""
    A = _as(A_bits, np.uint16)
    Bt = _as(Bt_bits, np.uint16)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    s = np.empty(rows.shape[0], dtype=np.float64)
    sa = np.empty(rows.shape[0], dtype=np.float64)
    m, k = A.shape
    n = Bt.shape[0]
    rc = _load().oracle_gemm_bf16_entries(m, k, n, _ptr(A), _ptr(Bt), rows.shape[0],
                                          _ptr(rows), _ptr(cols), _ptr(s), _ptr(sa))
    _check(rc)
    return s, sa


REQUANT_BF16 = 1
REQUANT_I8 = 2


def requant(C, row_scale, col_scale, out: str):
    """D = q((float(C) * row_scale[i]) * col_scale[j]) elementwise, every step
    one binary32 operation rounded to nearest even; q rounds to bfloat16
    (out = "bf16", returned as uint16 bit patterns) or to int8 with ties to
    even and saturation (out = "i8")."""
    C = _as(C, np.int32)
    rs = _as(row_scale, np.float32)
    cs = _as(col_scale, np.float32)
    m, n = C.shape
    if rs.shape != (m,) or cs.shape != (n,):
        raise ValueError("scale shapes")
    kind = {"bf16": REQUANT_BF16, "i8": REQUANT_I8}[out]
    D = np.empty((m, n), dtype=np.uint16 if kind == REQUANT_BF16 else np.int8)
    _check(_load().oracle_requant(m, n, _ptr(C), _ptr(rs), _ptr(cs), kind, _ptr(D)))
    return D
