#!/usr/bin/env python
"""Run one SDPA operation repeatedly on one synthetic case, for profilers (ncu) and quick
timing.  Every launch goes through the C ABI exactly as in normal use.

  python bench_profile.py --op fwd|bwd|step \\
      --B 2 --Hq 32 --Hkv 8 --L 4096 --D 128 --dtype bf16 --causal --iters 4 \\
      [--mask padding|additive]

--L is Lq (and Lkv unless --Lkv is given).  --mask padding passes a boolean key-padding
mask [B, 1, 1, Lkv] hiding the last 10% of the keys; --mask additive passes one N(0, 1)
[Lq, Lkv] mask in the element type, shared by every batch and head (seed 6).  Prints the
mean CUDA-event time per call (after one warm-up call).
"""
from __future__ import annotations

import argparse
import math
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

from scaled_dot_product_flash_gb300 import _lib, api  # noqa: E402
from scaled_dot_product_flash_gb300.inputs import Shape, draw  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", choices=["fwd", "bwd", "step"], default="fwd")
    ap.add_argument("--B", type=int, default=2)
    ap.add_argument("--Hq", type=int, default=32)
    ap.add_argument("--Hkv", type=int, default=8)
    ap.add_argument("--L", type=int, default=4096)
    ap.add_argument("--Lkv", type=int, default=None)
    ap.add_argument("--D", type=int, default=128)
    ap.add_argument("--dtype", default="bf16", choices=["f32", "f16", "bf16"])
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--path", default="auto", choices=["auto", "tensor", "simt", "vector"])
    ap.add_argument("--iters", type=int, default=4)
    ap.add_argument("--mask", default="none", choices=["none", "padding", "additive"])
    a = ap.parse_args()
    shape = Shape(a.B, a.Hq, a.Hkv, a.L, a.Lkv or a.L, a.D)
    q, k, v, do = (t.cuda() for t in draw(shape, 3, a.dtype))
    scale = 1.0 / math.sqrt(a.D)
    Lkv = a.Lkv or a.L
    mask = None
    if a.mask == "padding":
        mask = torch.ones(a.B, 1, 1, Lkv, dtype=torch.bool, device="cuda")
        mask[..., int(0.9 * Lkv):] = False
    elif a.mask == "additive":
        gen = torch.Generator(device="cpu").manual_seed(6)
        mask = torch.randn(a.L, Lkv, generator=gen).to(q.dtype).cuda()
    path = {"auto": _lib.PATH_AUTO, "tensor": _lib.PATH_TENSOR, "simt": _lib.PATH_SIMT,
            "vector": _lib.PATH_VECTOR}[a.path]
    with api.force_path(path):
        out, lse = api.attention_forward(q, k, v, scale=scale, is_causal=a.causal, attn_mask=mask)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(max(16, api.workspace_bytes(q, k)), device="cuda", dtype=torch.uint8)

        def once():
            if a.op in ("fwd", "step"):
                api.attention_forward(q, k, v, scale=scale, is_causal=a.causal, out=out, lse=lse,
                                      attn_mask=mask)
            if a.op in ("bwd", "step"):
                api.attention_backward(q, k, v, out, do, lse, scale=scale, is_causal=a.causal,
                                       workspace=ws, dq=dq, dk=dk, dv=dv, attn_mask=mask)

        once()
        api.poll_status()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(a.iters):
            once()
        e1.record()
        api.poll_status()
    ms = e0.elapsed_time(e1) / a.iters
    f = 4.0 * a.B * a.Hq * a.L * (a.Lkv or a.L) * a.D * (0.5 if a.causal else 1.0)
    mult = {"fwd": 1.0, "bwd": 2.5, "step": 3.5}[a.op]
    print(f"{a.op}: {ms:.4f} ms per call, {mult * f / ms / 1e9:.1f} TFLOP/s")


if __name__ == "__main__":
    main()
