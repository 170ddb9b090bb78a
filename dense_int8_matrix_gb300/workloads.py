"""Seeded synthetic inputs for the dense GEMM workloads.

This module only draws random numbers; it holds none of the GEMM's
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.
Every tensor is made on the CPU with a fresh ``torch.Generator`` seeded per
(workload, shape): A is drawn first, then Bt (B stored K-major, n x k).

Workloads (all sizes (m, k, n)):

* ``i8_256``     256^3, int8 uniform in [-128, 127], seed 0.  One tile the
  size of the TPU's 256x256 INT8 array.
* ``i8_4096``    4096^3, int8 uniform in [-128, 127], seed 1.
* ``i8_skinny``  m in {1, 8, 16, 32, 64, 128} x k = n = 8192.  A uniform in
  [-64, 63]; Bt = round-half-even(32 * N(0, 1)) clamped to [-128, 127];
  seed 2.
* ``i8_ragged``  (1000, 777, 3000), (4097, 16384, 255), (8192, 8192, 8192),
  int8 uniform in [-128, 127], seed 3.
* ``bf16_8192``  8192^3, N(0, 1) rounded to bf16 (round-to-nearest-even),
  fp32 output, seed 4.
"""

from __future__ import annotations

import hashlib

import torch

WORKLOADS = {
    "i8_256": {"dtype": "i8", "shapes": [(256, 256, 256)], "seed": 0,
               "a": ("uniform", -128, 127), "b": ("uniform", -128, 127)},
    "i8_4096": {"dtype": "i8", "shapes": [(4096, 4096, 4096)], "seed": 1,
                "a": ("uniform", -128, 127), "b": ("uniform", -128, 127)},
    "i8_skinny": {"dtype": "i8",
                  "shapes": [(m, 8192, 8192) for m in (1, 8, 16, 32, 64, 128)],
                  "seed": 2,
                  "a": ("uniform", -64, 63), "b": ("normal_clip", 32.0)},
    "i8_ragged": {"dtype": "i8",
                  "shapes": [(1000, 777, 3000), (4097, 16384, 255), (8192, 8192, 8192)],
                  "seed": 3,
                  "a": ("uniform", -128, 127), "b": ("uniform", -128, 127)},
    "bf16_8192": {"dtype": "bf16", "shapes": [(8192, 8192, 8192)], "seed": 4,
                  "a": ("normal_bf16",), "b": ("normal_bf16",)},
}


def _draw(spec, shape, gen: torch.Generator) -> torch.Tensor:
    kind = spec[0]
    if kind == "uniform":
        lo, hi = spec[1], spec[2]
        return torch.randint(lo, hi + 1, shape, generator=gen, dtype=torch.int8)
    if kind == "normal_clip":
        x = torch.randn(shape, generator=gen, dtype=torch.float32) * spec[1]
        return torch.round(x).clamp_(-128, 127).to(torch.int8)
    if kind == "normal_bf16":
        return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)
    raise ValueError(kind)


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def make_inputs(workload: str, shape, seed_offset: int = 0):
    """(A, Bt) CPU tensors for one shape of a named workload.

    ``seed_offset`` != 0 draws a further independent input set of the same
    distribution (used to rotate inputs through more memory than L2)."""
    spec = WORKLOADS[workload]
    m, k, n = shape
    g = generator(spec["seed"] + 1000003 * seed_offset)
    A = _draw(spec["a"], (m, k), g)
    Bt = _draw(spec["b"], (n, k), g)
    return A, Bt


def random_i8(shape, seed: int, lo: int = -128, hi: int = 127) -> torch.Tensor:
    return torch.randint(lo, hi + 1, tuple(shape), generator=generator(seed),
                         dtype=torch.int8)


def random_bf16(shape, seed: int, scale: float = 1.0) -> torch.Tensor:
    x = torch.randn(tuple(shape), generator=generator(seed), dtype=torch.float32)
    return (x * scale).to(torch.bfloat16)


def requant_scales(m: int, n: int, k: int, seed: int, c_std_per_sqrt_k: float = 5461.0, target: float = 40.0):
    """Seeded per-row and per-column fp32 scales for requantising an int32
    product of depth k: each drawn uniformly from [0.5, 1.5) times a base, so
    that their product times the typical |C| (c_std_per_sqrt_k * sqrt(k);
    5461 for int8 uniform in [-128, 127]) is about `target` (some int8
    results saturate, bfloat16 results span several binades)."""
    g = generator(seed)
    base = (target / (c_std_per_sqrt_k * float(k) ** 0.5)) ** 0.5
    rs = (torch.rand((m,), generator=g, dtype=torch.float32) + 0.5) * base
    cs = (torch.rand((n,), generator=g, dtype=torch.float32) + 0.5) * base
    return rs, cs


def shape_seed(tag: str) -> int:
    """A stable seed derived from a text tag (for test cases)."""
    return int.from_bytes(hashlib.sha256(tag.encode()).digest()[:4], "little")
