"""GB300-native dense GEMM: int8 x int8 -> int32 and bf16 x bf16 -> fp32.

The compute runs in the CUDA shared library ``libgemm_gb300.so`` built from
``csrc/`` for sm_103a; ``binding`` is a thin ctypes layer over its C ABI.
Importing this package does not load the library; the first binding call
does, and fails loudly if the library is missing.
"""

from __future__ import annotations

import importlib

__all__ = ["binding", "workloads"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module("." + name, __name__)
    raise AttributeError(name)
