"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws numbers and rounds them to the
requested element type.  The oracle receives the rounded values (upcast exactly), the
CUDA path receives the same values in the element type.

Recipe: ``numpy.random.default_rng(seed).standard_normal(shape, dtype=float32)`` drawn in
the order Q [B,Hq,Lq,D], K [B,Hkv,Lkv,D], V [B,Hkv,Lkv,D], dO [B,Hq,Lq,D], then rounded to
the element type with round-to-nearest-even.  This mirrors the timing script of the
PyTensor issue "PERF: detect scaled-dot-product-attention pattern and lower to
mx.fast.scaled_dot_product_attention" (section "Reproducer + metrics"), which draws
Q, K, V with ``default_rng(0).standard_normal`` at [B, H, S, hd].
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}


@dataclass(frozen=True)
class Shape:
    B: int
    Hq: int
    Hkv: int
    Lq: int
    Lkv: int
    D: int

    @property
    def q_shape(self):
        return (self.B, self.Hq, self.Lq, self.D)

    @property
    def kv_shape(self):
        return (self.B, self.Hkv, self.Lkv, self.D)


def draw(shape: Shape, seed: int, dtype: str, rng: np.random.Generator | None = None):
    """Draw (q, k, v, dout) as CPU torch tensors of ``dtype`` ('f32', 'f16', 'bf16').

    Pass ``rng`` to continue an existing stream (several sub-runs drawn one after the
    other from one seed); otherwise a fresh ``default_rng(seed)`` is used.
    """
    if rng is None:
        rng = np.random.default_rng(seed)
    t = DTYPES[dtype]
    out = []
    for shp in (shape.q_shape, shape.kv_shape, shape.kv_shape, shape.q_shape):
        x = rng.standard_normal(shp, dtype=np.float32)
        out.append(torch.from_numpy(x).to(t))
    return tuple(out)


def as_f64(x: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a CPU or GPU tensor (for the oracle and comparisons)."""
    return x.detach().to("cpu", torch.float64).numpy()
