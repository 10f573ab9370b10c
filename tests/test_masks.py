"""Attention masks: boolean (True keeps the key) and additive masks over [B, Hq, Lq, Lkv],
broadcast where a dimension has size 1, fused into every kernel family forward and
backward ("[Metal] Add Flash Attention VJP for training", section "Limitations", names
mask gradients among what the Metal backward leaves unfused; "mps-flash-sdpa 0.1.0",
section "When MFA Dispatches vs. Falls Back", hands every mask with a False entry back).
GPU results are compared element by element with the CPU oracle at the parity tolerances.

Masks are drawn from fixed seeds in five shapes: a random boolean mask per (batch, head)
keeping 70% of the keys, an additive N(0, 2²) mask per head with 20% −inf entries, a
per-batch key-padding mask, one additive [Lq, Lkv] mask shared by every batch and head,
and a sparse boolean mask keeping about three keys a row (the output of such a row rests
on a few weights).  The first two each hide one whole row (O = 0, lse = −inf, zero
gradients).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from parity_util import LSE_REL, O_TOL, check_grad
from scaled_dot_product_flash_gb300 import _lib, api, autograd
from scaled_dot_product_flash_gb300.inputs import DTYPES, Shape, as_f64, draw

pytestmark = pytest.mark.gpu


def make_mask(kind, shape, seed, dtype):
    """(CPU torch mask as passed to the GPU, the same values as the oracle's fp64 array)."""
    rng = np.random.default_rng(seed)
    B, Hq, Lq, Lkv = shape.B, shape.Hq, shape.Lq, shape.Lkv
    if kind == "bool":
        m = rng.random((B, Hq, Lq, Lkv)) < 0.7
        m[0, 0, min(3, Lq - 1)] = False
        t = torch.from_numpy(m)
        return t, m
    if kind == "sparse":
        # about three visible keys per row, spread over the KV tiles: the rows whose output
        # rests on a few weights, where rounding P to 16 bits shows most
        m = rng.random((B, Hq, Lq, Lkv)) < 3.0 / Lkv
        m[..., 0] |= ~m.any(axis=-1)
        return torch.from_numpy(m), m
    if kind == "padding":
        m = np.zeros((B, 1, 1, Lkv), dtype=bool)
        for b in range(B):
            m[b, :, :, :max(1, Lkv - 37 * (b + 1))] = True
        return torch.from_numpy(m), m
    if kind == "headrow":
        # one row per (batch, head), every query sees it: row stride 0, head stride nonzero
        m = rng.random((B, Hq, 1, Lkv)) < 0.8
        m[..., 0] = True
        return torch.from_numpy(m), m
    if kind == "addrow":
        m = (rng.standard_normal((1, Hq, 1, Lkv)) * 2.0).astype(np.float32)
        m[rng.random(m.shape) < 0.2] = -np.inf
        m[..., 0] = 0.0
    elif kind == "additive":
        m = (rng.standard_normal((1, Hq, Lq, Lkv)) * 2.0).astype(np.float32)
        m[rng.random(m.shape) < 0.2] = -np.inf
        m[0, Hq - 1, Lq // 2] = -np.inf
    elif kind == "shared":
        m = rng.standard_normal((Lq, Lkv)).astype(np.float32)
    else:
        raise KeyError(kind)
    t = torch.from_numpy(m).to(DTYPES[dtype])   # the element type the kernels read
    return t, as_f64(t)


def check_forward_masked(dtype, o, lse, o_ref, lse_ref, what=""):
    err_o = float(np.max(np.abs(o - o_ref)))
    assert err_o <= O_TOL[dtype], f"{what} O max-abs {err_o:.3e}"
    hidden = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), hidden), f"{what} rows with no visible key differ"
    seen = ~hidden
    if seen.any():
        err = np.abs(lse[seen] - lse_ref[seen]) / np.maximum(1.0, np.abs(lse_ref[seen]))
        assert float(err.max()) <= LSE_REL, f"{what} lse rel {float(err.max()):.3e}"


def run_case(shape, dtype, causal, kind, seed, path=_lib.PATH_AUTO, sinks=None):
    q, k, v, do = draw(shape, seed, dtype)
    mask_t, mask_n = make_mask(kind, shape, seed + 1, dtype)
    scale = 1.0 / math.sqrt(shape.D)
    with api.force_path(path):
        qd, kd, vd, dod, md = (t.cuda() for t in (q, k, v, do, mask_t))
        sd = sinks.cuda() if sinks is not None else None
        o, lse = api.attention_forward(qd, kd, vd, scale=scale, is_causal=causal, sinks=sd,
                                       attn_mask=md)
        g = api.attention_backward(qd, kd, vd, o, dod, lse, scale=scale, is_causal=causal,
                                   sinks=sd, attn_mask=md)
        api.poll_status()
    qn, kn, vn, don = (as_f64(t) for t in (q, k, v, do))
    sn = as_f64(sinks) if sinks is not None else None
    what = f"{shape} {dtype} causal={causal} {kind}"
    o_ref, lse_ref = oracle.sdpa_forward(qn, kn, vn, scale, causal, sinks=sn, mask=mask_n)
    check_forward_masked(dtype, as_f64(o), as_f64(lse), o_ref, lse_ref, what)
    refs = oracle.sdpa_backward(qn, kn, vn, don, scale, causal, sinks=sn, mask=mask_n)
    for name, got, ref in zip(("dq", "dk", "dv"), g[:3], refs[:3]):
        check_grad(dtype, name, as_f64(got), ref, what)
    return g, refs


CASES = [
    (Shape(2, 8, 2, 200, 200, 128), "bf16", False, _lib.PATH_AUTO, "bool"),      # tensor cores
    (Shape(1, 4, 4, 96, 160, 64), "f16", False, _lib.PATH_AUTO, "additive"),     # tensor cores
    (Shape(1, 4, 2, 150, 300, 96), "bf16", 2, _lib.PATH_AUTO, "padding"),        # D = 96, bottom-right
    (Shape(1, 4, 1, 130, 260, 32), "f16", True, _lib.PATH_AUTO, "shared"),       # D = 32, causal
    (Shape(1, 4, 2, 40, 70, 32), "f32", True, _lib.PATH_AUTO, "bool"),           # CUDA cores
    (Shape(1, 4, 2, 130, 130, 64), "bf16", False, _lib.PATH_SIMT, "additive"),   # forced CUDA cores
    (Shape(2, 8, 2, 4, 300, 128), "bf16", False, _lib.PATH_AUTO, "bool"),        # short query, MMA
    (Shape(2, 8, 2, 4, 300, 64), "bf16", True, _lib.PATH_AUTO, "shared"),        # short query, MMA, D = 64
    (Shape(1, 4, 2, 5, 90, 96), "f32", False, _lib.PATH_AUTO, "additive"),       # short query, CUDA cores
    (Shape(3, 4, 4, 1, 77, 64), "f16", False, _lib.PATH_AUTO, "padding"),        # single query row
    (Shape(1, 4, 2, 50, 77, 256), "f16", False, _lib.PATH_AUTO, "additive"),     # D = 256 on tensor cores
    (Shape(1, 4, 2, 200, 330, 256), "bf16", True, _lib.PATH_AUTO, "bool"),       # D = 256, several KV tiles
    (Shape(1, 4, 2, 200, 330, 256), "f16", 2, _lib.PATH_TENSOR, "padding"),      # D = 256 forced, one row, bottom-right
    (Shape(2, 4, 4, 70, 200, 256), "bf16", True, _lib.PATH_TENSOR, "shared"),    # D = 256 forced, one mask for all
    (Shape(1, 4, 1, 129, 150, 256), "bf16", False, _lib.PATH_TENSOR, "additive"),  # D = 256 forced, G = 4
    (Shape(1, 4, 2, 50, 77, 256), "f32", False, _lib.PATH_AUTO, "padding"),      # D = 256, CUDA cores
    (Shape(2, 4, 2, 260, 520, 128), "bf16", False, _lib.PATH_AUTO, "sparse"),    # few keys a row, MMA
    (Shape(1, 4, 2, 130, 400, 256), "bf16", False, _lib.PATH_AUTO, "sparse"),    # few keys a row, D = 256
    # one mask row for every query (row stride 0): dK/dV reads it per key, no mask tile
    (Shape(2, 4, 2, 300, 300, 128), "bf16", False, _lib.PATH_AUTO, "padding"),   # key padding, D = 128
    (Shape(2, 8, 2, 200, 330, 128), "bf16", True, _lib.PATH_AUTO, "headrow"),    # one row per head
    (Shape(1, 4, 1, 150, 260, 64), "f16", False, _lib.PATH_AUTO, "addrow"),      # additive row, G = 4
    (Shape(1, 4, 2, 130, 200, 256), "bf16", True, _lib.PATH_AUTO, "headrow"),    # D = 256
]


@pytest.mark.parametrize("shape,dtype,causal,path,kind", CASES)
def test_masks_match_oracle(shape, dtype, causal, path, kind):
    run_case(shape, dtype, causal, kind, 121, path)


def test_mask_with_sinks_and_causal():
    shape = Shape(2, 8, 2, 200, 200, 128)
    sinks = torch.from_numpy(np.random.default_rng(123).standard_normal(8).astype(np.float32) + 3)
    g, refs = run_case(shape, "bf16", True, "additive", 124, sinks=sinks)
    from parity_util import rel_frob
    assert rel_frob(as_f64(g[3]), refs[3]) <= 1e-2


@pytest.mark.parametrize("shape,dtype,path", [
    (Shape(1, 4, 4, 96, 160, 64), "f16", _lib.PATH_AUTO),      # tensor cores
    (Shape(1, 4, 2, 40, 70, 32), "f32", _lib.PATH_AUTO),       # CUDA cores
    (Shape(2, 4, 2, 4, 300, 128), "bf16", _lib.PATH_AUTO),     # short query
])
def test_minus_infinity_sink_on_a_row_that_sees_no_key(shape, dtype, path):
    """The additive mask hides one whole row of the last head, whose sink is −inf (no
    sink): that head's sink gradient is exactly 0 and every sink gradient is finite and
    matches the oracle."""
    sinks = torch.tensor([2.5, -1.0, 0.5, -np.inf], dtype=torch.float32)
    g, refs = run_case(shape, dtype, False, "additive", 131, path, sinks=sinks)
    got = as_f64(g[3])
    assert np.all(np.isfinite(got)), got
    assert got[-1] == 0.0
    if dtype == "f32":
        assert float(np.max(np.abs(got - refs[3]))) <= 1e-4
    else:
        from parity_util import rel_frob
        assert rel_frob(got, refs[3]) <= 1e-2


@pytest.mark.parametrize("shape,dtype", [
    (Shape(1, 4, 2, 300, 384, 128), "bf16"),   # D = 128: Q tile 1 of the first block hidden
    (Shape(1, 2, 1, 260, 300, 256), "f16"),    # D = 256
])
def test_mask_hiding_whole_query_tiles(shape, dtype):
    """A boolean mask per (batch, head) that hides every key of query rows [128, 256) (a
    whole 128-row Q tile) of the first head and keeps a random 70% elsewhere: those rows
    give O = 0, lse = −inf and zero dQ, and everything matches the oracle."""
    rng = np.random.default_rng(140)
    m = rng.random((shape.B, shape.Hq, shape.Lq, shape.Lkv)) < 0.7
    m[:, 0, 128:256, :] = False
    q, k, v, do = draw(shape, 141, dtype)
    scale = 1.0 / math.sqrt(shape.D)
    qd, kd, vd, dod, md = (t.cuda() for t in (q, k, v, do, torch.from_numpy(m)))
    o, lse = api.attention_forward(qd, kd, vd, scale=scale, attn_mask=md)
    g = api.attention_backward(qd, kd, vd, o, dod, lse, scale=scale, attn_mask=md)
    api.poll_status()
    qn, kn, vn, don = (as_f64(t) for t in (q, k, v, do))
    o_ref, lse_ref = oracle.sdpa_forward(qn, kn, vn, scale, False, mask=m)
    check_forward_masked(dtype, as_f64(o), as_f64(lse), o_ref, lse_ref, "whole tiles")
    assert np.all(as_f64(o)[:, 0, 128:256] == 0.0)
    assert np.all(np.isneginf(as_f64(lse)[:, 0, 128:256]))
    assert np.all(as_f64(g[0])[:, 0, 128:256] == 0.0)
    refs = oracle.sdpa_backward(qn, kn, vn, don, scale, False, mask=m)
    for name, got, ref in zip(("dq", "dk", "dv"), g[:3], refs[:3]):
        check_grad(dtype, name, as_f64(got), ref, "whole tiles")


def test_masked_autograd_matches_oracle():
    shape = Shape(1, 8, 2, 160, 224, 128)
    q, k, v, do = draw(shape, 125, "bf16")
    mask_t, mask_n = make_mask("bool", shape, 126, "bf16")
    qd, kd, vd = (t.cuda().requires_grad_(True) for t in (q, k, v))
    out = autograd.scaled_dot_product_attention(qd, kd, vd, attn_mask=mask_t.cuda(),
                                                enable_gqa=True)
    out.backward(do.cuda())
    torch.cuda.synchronize()
    scale = 1.0 / math.sqrt(shape.D)
    qn, kn, vn, don = (as_f64(t) for t in (q, k, v, do))
    o_ref, _ = oracle.sdpa_forward(qn, kn, vn, scale, False, mask=mask_n)
    assert float(np.max(np.abs(as_f64(out.detach()) - o_ref))) <= O_TOL["bf16"]
    refs = oracle.sdpa_backward(qn, kn, vn, don, scale, False, mask=mask_n)
    for name, leaf, ref in zip(("dq", "dk", "dv"), (qd, kd, vd), refs):
        check_grad("bf16", name, as_f64(leaf.grad), ref, "autograd mask")


def test_banded_mask_at_a_larger_size():
    """Headline-like shape (GQA 4, D = 128, 2048 rows) with one [Lq, Lkv] additive mask
    shared by every head: a band of 512 keys around the diagonal (−inf outside) with
    N(0, 1) values inside.  The oracle recomputes sampled rows of four heads and the full
    backward of KV group 0."""
    shape = Shape(1, 8, 2, 2048, 2048, 128)
    q, k, v, do = draw(shape, 127, "bf16")
    rng = np.random.default_rng(128)
    m = rng.standard_normal((2048, 2048)).astype(np.float32)
    ii, jj = np.indices(m.shape)
    m[np.abs(ii - jj) > 256] = -np.inf
    mask_t = torch.from_numpy(m).to(torch.bfloat16)
    mask_n = as_f64(mask_t)
    scale = 1.0 / math.sqrt(shape.D)
    qd, kd, vd, dod, md = (t.cuda() for t in (q, k, v, do, mask_t))
    o, lse = api.attention_forward(qd, kd, vd, scale=scale, attn_mask=md)
    dq, dk, dv = api.attention_backward(qd, kd, vd, o, dod, lse, scale=scale, attn_mask=md)
    api.poll_status()
    rows = np.array([0, 1, 255, 256, 1000, 2047])
    G = shape.Hq // shape.Hkv
    for h in (0, 3, 4, 7):
        o_ref, lse_ref = oracle.head_forward(as_f64(q[0, h]), as_f64(k[0, h // G]),
                                             as_f64(v[0, h // G]), scale, False, rows=rows,
                                             mask=mask_n)
        check_forward_masked("bf16", as_f64(o[0, h])[rows], as_f64(lse[0, h])[rows], o_ref,
                             lse_ref, f"h={h}")
    dq_ref, dk_ref, dv_ref = oracle.group_backward(as_f64(q), as_f64(k), as_f64(v), as_f64(do),
                                                   scale, False, 0, 0, row_block=512,
                                                   mask=mask_n)
    check_grad("bf16", "dq", as_f64(dq[0, :G]), dq_ref, "banded")
    check_grad("bf16", "dk", as_f64(dk[0, 0]), dk_ref, "banded")
    check_grad("bf16", "dv", as_f64(dv[0, 0]), dv_ref, "banded")
