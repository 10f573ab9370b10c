"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and compare it
with the CPU oracle on the same seeded inputs, at the tolerances the target states.

Tolerances (per element type):
  fp32      : max |O - O_ref| <= 1e-5 ; max |dX - dX_ref| <= 1e-4 for dQ, dK, dV
  fp16      : max |O - O_ref| <= 2e-3 ; ||dX - dX_ref||_F / ||dX_ref||_F <= 1e-2
  bf16      : max |O - O_ref| <= 8e-3 ; same relative Frobenius bound on gradients
  logsumexp : |lse - lse_ref| <= 1e-4 · max(1, |lse_ref|)   (all types)
The max(1, ·) floor reads "1e-4 relative" so that it stays meaningful where the
logsumexp itself is near zero (e.g. the first causal row, where it is one score).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from scaled_dot_product_flash_gb300 import api
from scaled_dot_product_flash_gb300.inputs import Shape, as_f64, draw

O_TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 8e-3}
GRAD_ABS_F32 = 1e-4
GRAD_REL_FROB = 1e-2
LSE_REL = 1e-4


def run_gpu(q, k, v, do, scale, causal, backward=True):
    """Forward (+ backward) on the GPU through the C ABI; returns CPU float64 arrays."""
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev).contiguous() for t in (q, k, v, do))
    out, lse = api.attention_forward(qd, kd, vd, scale=scale, is_causal=causal)
    res = {"o": out, "lse": lse}
    if backward:
        dq, dk, dv = api.attention_backward(qd, kd, vd, out, dod, lse, scale=scale,
                                            is_causal=causal)
        res.update(dq=dq, dk=dk, dv=dv)
    api.poll_status()
    return {n: as_f64(t) for n, t in res.items()}


def rel_frob(a, ref):
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(a - ref) / (den if den > 0 else 1.0))


def check_forward(dtype, o, lse, o_ref, lse_ref, what=""):
    err_o = float(np.max(np.abs(o - o_ref))) if o.size else 0.0
    assert err_o <= O_TOL[dtype], f"{what} O max-abs {err_o:.3e} > {O_TOL[dtype]}"
    err_l = np.abs(lse - lse_ref) / np.maximum(1.0, np.abs(lse_ref))
    assert float(err_l.max()) <= LSE_REL, f"{what} lse rel {float(err_l.max()):.3e}"
    return err_o, float(err_l.max())


def check_grad(dtype, name, g, g_ref, what=""):
    if dtype == "f32":
        err = float(np.max(np.abs(g - g_ref)))
        assert err <= GRAD_ABS_F32, f"{what} {name} max-abs {err:.3e} > {GRAD_ABS_F32}"
    else:
        err = rel_frob(g, g_ref)
        assert err <= GRAD_REL_FROB, f"{what} {name} rel-Frobenius {err:.3e} > {GRAD_REL_FROB}"
    return err


def full_parity(shape: Shape, dtype: str, causal: bool, seed: int, scale=None,
                backward=True, inputs=None):
    """Every output element compared with the oracle (sizes the oracle runs in seconds)."""
    scale = 1.0 / math.sqrt(shape.D) if scale is None else scale
    q, k, v, do = inputs if inputs is not None else draw(shape, seed, dtype)
    got = run_gpu(q, k, v, do, scale, causal, backward)
    qn, kn, vn, don = (as_f64(t) for t in (q, k, v, do))
    o_ref, lse_ref = oracle.sdpa_forward(qn, kn, vn, scale, causal)
    what = f"{shape} {dtype} causal={causal}"
    errs = {}
    errs["o"], errs["lse"] = check_forward(dtype, got["o"], got["lse"], o_ref, lse_ref, what)
    if backward:
        dq_ref, dk_ref, dv_ref = oracle.sdpa_backward(qn, kn, vn, don, scale, causal)
        for n, ref in (("dq", dq_ref), ("dk", dk_ref), ("dv", dv_ref)):
            errs[n] = check_grad(dtype, n, got[n], ref, what)
    return errs


def sampled_parity(shape: Shape, dtype: str, causal: bool, seed: int, groups, scale=None,
                   row_block=1024):
    """Full-size run on the GPU; the oracle recomputes whole (batch, KV-head) groups.

    For each sampled (b, g) the oracle produces O and lse of the G query heads, dQ of
    those heads, and dK, dV of KV head g; those are compared element by element.
    """
    scale = 1.0 / math.sqrt(shape.D) if scale is None else scale
    q, k, v, do = draw(shape, seed, dtype)
    got = run_gpu(q, k, v, do, scale, causal, True)
    G = shape.Hq // shape.Hkv
    errs = []
    for b, g in groups:
        heads = range(g * G, (g + 1) * G)
        kg, vg = as_f64(k[b, g]), as_f64(v[b, g])
        for h in heads:
            o_ref, lse_ref = oracle.head_forward(as_f64(q[b, h]), kg, vg, scale, causal,
                                                 row_block=row_block)
            check_forward(dtype, got["o"][b, h], got["lse"][b, h], o_ref, lse_ref,
                          f"b={b} h={h}")
        qs = as_f64(q[b:b + 1])
        dos = as_f64(do[b:b + 1])
        dq_ref, dk_ref, dv_ref = oracle.group_backward(
            qs, as_f64(k[b:b + 1]), as_f64(v[b:b + 1]), dos, scale, causal, 0, g,
            row_block=row_block)
        e = {
            "dq": check_grad(dtype, "dq", got["dq"][b, g * G:(g + 1) * G], dq_ref),
            "dk": check_grad(dtype, "dk", got["dk"][b, g], dk_ref),
            "dv": check_grad(dtype, "dv", got["dv"][b, g], dv_ref),
        }
        errs.append(e)
    return errs
