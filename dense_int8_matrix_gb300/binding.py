"""ctypes binding of libgemm_gb300.so (include/dense_int8_matrix.h).

Argument marshalling only: every step of the GEMM runs in the library's CUDA
kernels.  Functions carry the C names.  Device buffers may be passed as
torch CUDA tensors (checked for dtype, shape, contiguity and device) or as
raw integer addresses.  If the library is missing, the first call raises;
there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

from . import build as _build

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_MISALIGNED = 2
GEMM_ERR_UNSUPPORTED_DEVICE = 3
GEMM_ERR_CUDA = 4
GEMM_ERR_OVERFLOW_RISK = 5
GEMM_ERR_TIMEOUT = 6

GEMM_PATH_TENSOR = 0
GEMM_PATH_SKINNY = 1
GEMM_DTYPE_I8 = 0
GEMM_DTYPE_BF16 = 1
GEMM_KERNEL_STAGE = 0
GEMM_KERNEL_TC = 1
GEMM_KERNEL_SKINNY = 2
GEMM_KERNEL_REQUANT = 3
GEMM_KERNEL_KINDS = 4
GEMM_OUT_BF16 = 1
GEMM_OUT_I8 = 2
GEMM_PLAN_VERSION = 2
GEMM_I8_MAX_K = 131071
GEMM_NOALLOC_SCRATCH_BYTES = 64 << 20

# every function the header declares
EXPORTED = (
    "gemm_i8_plan", "gemm_bf16_plan", "gemm_plan_for_sms", "gemm_i8_run", "gemm_bf16_run",
    "gemm_i8_run_host", "gemm_bf16_run_host", "gemm_device_error", "gemm_trace_begin",
    "gemm_trace_collect", "gemm_tc_kernel_info", "gemm_selftest_wait_timeout", "gemm_status_string",
    "gemm_i8_run_noalloc", "gemm_pool_usage", "gemm_i8_run_requant",
)


class gemm_plan(ctypes.Structure):
    _fields_ = [
        ("version", ctypes.c_int32), ("path", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("num_sms", ctypes.c_int32),
        ("m", ctypes.c_int64), ("k", ctypes.c_int64), ("n", ctypes.c_int64),
        ("bm", ctypes.c_int32), ("bn", ctypes.c_int32), ("bk", ctypes.c_int32),
        ("stages", ctypes.c_int32), ("tiles", ctypes.c_int32), ("bpc", ctypes.c_int32),
        ("grid", ctypes.c_int32), ("waves", ctypes.c_int32), ("k_pitch", ctypes.c_int32),
        ("chunk_k", ctypes.c_int32), ("fallback", ctypes.c_int32), ("split_k", ctypes.c_int32),
        ("ratio", ctypes.c_double), ("workspace_bytes", ctypes.c_int64),
        ("split_from", ctypes.c_int32), ("a_on_chip", ctypes.c_int32),
        ("reserved", ctypes.c_int64 * 3),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_
                if not name.startswith("reserved")}


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, _status_name(status)))


_lib = None


def _status_name(s: int) -> str:
    names = {0: "GEMM_OK", 1: "GEMM_ERR_INVALID_ARG", 2: "GEMM_ERR_MISALIGNED",
             3: "GEMM_ERR_UNSUPPORTED_DEVICE", 4: "GEMM_ERR_CUDA", 5: "GEMM_ERR_OVERFLOW_RISK",
             6: "GEMM_ERR_TIMEOUT"}
    return names.get(s, "status %d" % s)


def library_path() -> str:
    return _build.LIB_PATH


def load():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError("%s is not built (run __graft_entry__.build()); "
                           "the GEMM has no CPU fallback" % path)
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(gemm_plan)
    i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    sig = {
        "gemm_i8_plan": [i64, i64, i64, P],
        "gemm_bf16_plan": [i64, i64, i64, P],
        "gemm_plan_for_sms": [i32, i64, i64, i64, i32, P],
        "gemm_i8_run": [P, vp, vp, vp, vp],
        "gemm_bf16_run": [P, vp, vp, vp, vp],
        "gemm_i8_run_host": [P, vp, vp, vp, vp],
        "gemm_bf16_run_host": [P, vp, vp, vp, vp],
        "gemm_device_error": [vp, ctypes.POINTER(i32)],
        "gemm_trace_begin": [i32, i32],
        "gemm_trace_collect": [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(i32), ctypes.POINTER(i32)],
        "gemm_tc_kernel_info": [i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)],
        "gemm_selftest_wait_timeout": [i32, vp],
        "gemm_i8_run_noalloc": [P, vp, vp, vp, vp],
        "gemm_pool_usage": [ctypes.POINTER(i64), ctypes.POINTER(i64), i32],
        "gemm_i8_run_requant": [P, vp, vp, vp, vp, i32, vp, vp],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.gemm_status_string.argtypes = [ctypes.c_int]
    lib.gemm_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def gemm_status_string(status: int) -> str:
    return load().gemm_status_string(status).decode()


def _check(status: int, where: str):
    if status != GEMM_OK:
        raise GemmError(status, where)


# ------------------------------------------------------------------ plans --

def gemm_i8_plan(m: int, k: int, n: int) -> gemm_plan:
    p = gemm_plan()
    _check(load().gemm_i8_plan(m, k, n, ctypes.byref(p)), "gemm_i8_plan")
    return p


def gemm_bf16_plan(m: int, k: int, n: int) -> gemm_plan:
    p = gemm_plan()
    _check(load().gemm_bf16_plan(m, k, n, ctypes.byref(p)), "gemm_bf16_plan")
    return p


def gemm_plan_for_sms(dtype: int, m: int, k: int, n: int, num_sms: int) -> gemm_plan:
    p = gemm_plan()
    _check(load().gemm_plan_for_sms(dtype, m, k, n, num_sms, ctypes.byref(p)), "gemm_plan_for_sms")
    return p


# -------------------------------------------------------------------- run --

def _addr(x, dtype=None, shape=None, device=True):
    """Address of a tensor (after checks) or an integer address as is."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    import torch
    if not isinstance(x, torch.Tensor):
        raise TypeError("expected a torch tensor or an integer address")
    if dtype is not None and x.dtype != dtype:
        raise TypeError("expected %s, got %s" % (dtype, x.dtype))
    if shape is not None and tuple(x.shape) != tuple(shape):
        raise ValueError("expected shape %s, got %s" % (tuple(shape), tuple(x.shape)))
    if not x.is_contiguous():
        raise ValueError("tensor must be contiguous")
    if device and not x.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not device and x.is_cuda:
        raise ValueError("tensor must be in host memory")
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def gemm_i8_run(plan: gemm_plan, A, Bt, C, stream=None) -> None:
    import torch
    m, k, n = plan.m, plan.k, plan.n
    st = load().gemm_i8_run(ctypes.byref(plan), _addr(A, torch.int8, (m, k)), _addr(Bt, torch.int8, (n, k)),
                            _addr(C, torch.int32, (m, n)), _stream(stream))
    _check(st, "gemm_i8_run")


def gemm_bf16_run(plan: gemm_plan, A, Bt, C, stream=None) -> None:
    import torch
    m, k, n = plan.m, plan.k, plan.n
    st = load().gemm_bf16_run(ctypes.byref(plan), _addr(A, torch.bfloat16, (m, k)),
                              _addr(Bt, torch.bfloat16, (n, k)), _addr(C, torch.float32, (m, n)),
                              _stream(stream))
    _check(st, "gemm_bf16_run")


def gemm_i8_run_noalloc(plan: gemm_plan, A, Bt, C, stream=None) -> None:
    """gemm_i8_run without device allocation (fixed 64 MiB static scratch)."""
    import torch
    m, k, n = plan.m, plan.k, plan.n
    st = load().gemm_i8_run_noalloc(ctypes.byref(plan), _addr(A, torch.int8, (m, k)),
                                    _addr(Bt, torch.int8, (n, k)), _addr(C, torch.int32, (m, n)),
                                    _stream(stream))
    _check(st, "gemm_i8_run_noalloc")


def gemm_i8_run_requant(plan: gemm_plan, A, Bt, row_scale, col_scale, D, out_type=None, stream=None) -> None:
    """D = q((float(A x B) * row_scale[i]) * col_scale[j]) with q = bfloat16
    (D a torch.bfloat16 tensor) or saturated int8 (D a torch.int8 tensor)."""
    import torch
    m, k, n = plan.m, plan.k, plan.n
    if out_type is None:
        out_type = GEMM_OUT_BF16 if isinstance(D, torch.Tensor) and D.dtype == torch.bfloat16 else GEMM_OUT_I8
    d_dtype = torch.bfloat16 if out_type == GEMM_OUT_BF16 else torch.int8
    st = load().gemm_i8_run_requant(ctypes.byref(plan), _addr(A, torch.int8, (m, k)), _addr(Bt, torch.int8, (n, k)),
                                    _addr(row_scale, torch.float32, (m,)), _addr(col_scale, torch.float32, (n,)),
                                    out_type, _addr(D, d_dtype, (m, n)), _stream(stream))
    _check(st, "gemm_i8_run_requant")


def gemm_i8_run_host(plan: gemm_plan, A, Bt, C, stream=None) -> None:
    import torch
    m, k, n = plan.m, plan.k, plan.n
    st = load().gemm_i8_run_host(ctypes.byref(plan), _addr(A, torch.int8, (m, k), device=False),
                                 _addr(Bt, torch.int8, (n, k), device=False),
                                 _addr(C, torch.int32, (m, n), device=False), _stream(stream))
    _check(st, "gemm_i8_run_host")


def gemm_bf16_run_host(plan: gemm_plan, A, Bt, C, stream=None) -> None:
    import torch
    m, k, n = plan.m, plan.k, plan.n
    st = load().gemm_bf16_run_host(ctypes.byref(plan), _addr(A, torch.bfloat16, (m, k), device=False),
                                   _addr(Bt, torch.bfloat16, (n, k), device=False),
                                   _addr(C, torch.float32, (m, n), device=False), _stream(stream))
    _check(st, "gemm_bf16_run_host")


def gemm_device_error(stream=None):
    """(status, code): GEMM_OK or GEMM_ERR_TIMEOUT with the stage that gave up."""
    code = ctypes.c_int32(0)
    st = load().gemm_device_error(_stream(stream), ctypes.byref(code))
    return st, code.value


def gemm_pool_usage(reset_high: bool = False):
    """(bytes the library's pool holds, most bytes in use at once since the
    last reset); reset_high restarts the second from the current use."""
    reserved = ctypes.c_int64(0)
    high = ctypes.c_int64(0)
    _check(load().gemm_pool_usage(ctypes.byref(reserved), ctypes.byref(high), 1 if reset_high else 0),
           "gemm_pool_usage")
    return reserved.value, high.value


def gemm_trace_begin(capacity: int, every: int = 1) -> None:
    _check(load().gemm_trace_begin(capacity, every), "gemm_trace_begin")


def gemm_trace_collect():
    """Per kind: (summed ms of the timed units, timed units, launches counted)."""
    ms = (ctypes.c_float * GEMM_KERNEL_KINDS)()
    timed = (ctypes.c_int32 * GEMM_KERNEL_KINDS)()
    cnt = (ctypes.c_int32 * GEMM_KERNEL_KINDS)()
    _check(load().gemm_trace_collect(ms, timed, cnt), "gemm_trace_collect")
    return list(ms), list(timed), list(cnt)


def gemm_tc_kernel_info(bm: int, bn: int, dtype: int):
    regs = ctypes.c_int32(0)
    occ = ctypes.c_int32(0)
    _check(load().gemm_tc_kernel_info(bm, bn, dtype, ctypes.byref(regs), ctypes.byref(occ)),
           "gemm_tc_kernel_info")
    return regs.value, occ.value


def gemm_selftest_wait_timeout(timeout_us: int, stream=None) -> None:
    _check(load().gemm_selftest_wait_timeout(timeout_us, _stream(stream)), "gemm_selftest_wait_timeout")


# ------------------------------------------------------------ convenience --

def matmul_i8(A, Bt, out=None, stream=None):
    """int32 C = A x B for int8 CUDA tensors A (m x k) and Bt (n x k)."""
    import torch
    m, k = A.shape
    n = Bt.shape[0]
    plan = gemm_i8_plan(m, k, n)
    if out is None:
        out = torch.empty((m, n), dtype=torch.int32, device=A.device)
    gemm_i8_run(plan, A, Bt, out, stream)
    return out


def matmul_bf16(A, Bt, out=None, stream=None):
    """fp32 C = A x B for bf16 CUDA tensors A (m x k) and Bt (n x k)."""
    import torch
    m, k = A.shape
    n = Bt.shape[0]
    plan = gemm_bf16_plan(m, k, n)
    if out is None:
        out = torch.empty((m, n), dtype=torch.float32, device=A.device)
    gemm_bf16_run(plan, A, Bt, out, stream)
    return out
