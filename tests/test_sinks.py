"""Attention sinks: one learned logit per query head that joins every row's softmax as an
entry with a zero value vector ("[Metal] Add Flash Attention VJP for training", section
"Limitations", names sink gradients among what the Metal backward leaves unfused; here
they are fused).  GPU results are compared element by element with the CPU oracle at the
parity tolerances, in every kernel family, and the sink gradient with the oracle's.

Sink logits are drawn per head from a fixed seed: a normal spread around the size of a
row's logsumexp (so that the sink takes a visible share of each row), with one head at a
large value (the sink dominates) and one at −inf (no sink) where there are enough heads.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from parity_util import GRAD_ABS_F32, GRAD_REL_FROB, check_forward, check_grad, rel_frob
from scaled_dot_product_flash_gb300 import _lib, api, autograd
from scaled_dot_product_flash_gb300.inputs import Shape, as_f64, draw

pytestmark = pytest.mark.gpu


def draw_sinks(Hq, seed):
    rng = np.random.default_rng(seed)
    s = (rng.standard_normal(Hq) * 2.0 + 3.0).astype(np.float32)
    if Hq >= 4:
        s[1] = np.float32(12.0)
        s[2] = np.float32(-np.inf)
    return torch.from_numpy(s)


def check_dsinks(dtype, got, ref, what=""):
    if dtype == "f32":
        err = float(np.max(np.abs(got - ref)))
        assert err <= GRAD_ABS_F32, f"{what} dsinks max-abs {err:.3e}"
    else:
        err = rel_frob(got, ref)
        assert err <= GRAD_REL_FROB, f"{what} dsinks rel-Frobenius {err:.3e}"
    return err


CASES = [
    (Shape(2, 8, 2, 200, 200, 128), "bf16", True, _lib.PATH_AUTO),      # tensor cores, GQA, tail
    (Shape(1, 4, 4, 96, 160, 64), "f16", False, _lib.PATH_AUTO),        # tensor cores, Lq != Lkv
    (Shape(1, 4, 2, 150, 300, 96), "bf16", 2, _lib.PATH_AUTO),          # tensor cores, D = 96, bottom-right
    (Shape(1, 4, 1, 130, 260, 32), "f16", True, _lib.PATH_AUTO),        # tensor cores, D = 32
    (Shape(1, 4, 2, 40, 70, 32), "f32", True, _lib.PATH_AUTO),          # CUDA cores
    (Shape(1, 4, 2, 130, 130, 64), "bf16", True, _lib.PATH_SIMT),       # forced CUDA cores, bf16
    (Shape(2, 8, 2, 4, 300, 128), "bf16", False, _lib.PATH_AUTO),       # short query, warp MMA
    (Shape(1, 4, 2, 5, 90, 96), "f32", 2, _lib.PATH_AUTO),              # short query, CUDA cores
    (Shape(3, 4, 4, 1, 77, 64), "f16", False, _lib.PATH_AUTO),          # single query row
    (Shape(1, 4, 2, 40, 70, 256), "bf16", True, _lib.PATH_AUTO),        # D = 256: tensor-core forward
    (Shape(1, 4, 2, 40, 70, 256), "f32", True, _lib.PATH_AUTO),         # D = 256, CUDA cores
    (Shape(1, 4, 1, 300, 420, 256), "f16", False, _lib.PATH_AUTO),      # D = 256, several KV tiles
]


@pytest.mark.parametrize("shape,dtype,causal,path", CASES)
def test_sinks_match_oracle(shape, dtype, causal, path):
    q, k, v, do = draw(shape, 101, dtype)
    sinks = draw_sinks(shape.Hq, 102)
    scale = 1.0 / math.sqrt(shape.D)
    with api.force_path(path):
        qd, kd, vd, dod, sd = (t.cuda() for t in (q, k, v, do, sinks))
        o, lse = api.attention_forward(qd, kd, vd, scale=scale, is_causal=causal, sinks=sd)
        dq, dk, dv, ds = api.attention_backward(qd, kd, vd, o, dod, lse, scale=scale,
                                                is_causal=causal, sinks=sd)
        api.poll_status()
    qn, kn, vn, don = (as_f64(t) for t in (q, k, v, do))
    sn = as_f64(sinks)
    what = f"{shape} {dtype} causal={causal} path={path}"
    o_ref, lse_ref = oracle.sdpa_forward(qn, kn, vn, scale, causal, sinks=sn)
    check_forward(dtype, as_f64(o), as_f64(lse), o_ref, lse_ref, what)
    refs = oracle.sdpa_backward(qn, kn, vn, don, scale, causal, sinks=sn)
    for name, g, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs[:3]):
        check_grad(dtype, name, as_f64(g), ref, what)
    check_dsinks(dtype, as_f64(ds), refs[3], what)


@pytest.mark.parametrize("shape,dtype,causal", [
    (Shape(2, 8, 2, 200, 200, 128), "bf16", True),
    (Shape(1, 4, 2, 40, 70, 64), "f32", False),
    (Shape(2, 8, 2, 4, 300, 128), "bf16", True),
])
def test_minus_infinity_sinks_are_bitwise_no_sinks(shape, dtype, causal):
    """exp2(−inf) = 0 is added to each row sum and the output factor stays 1: the results
    are the same bits as without sinks, and the sink gradients are exactly zero."""
    q, k, v, do = (t.cuda() for t in draw(shape, 103, dtype))
    sinks = torch.full((shape.Hq,), -math.inf, device="cuda")
    o0, l0 = api.attention_forward(q, k, v, is_causal=causal)
    g0 = api.attention_backward(q, k, v, o0, do, l0, is_causal=causal)
    o1, l1 = api.attention_forward(q, k, v, is_causal=causal, sinks=sinks)
    g1 = api.attention_backward(q, k, v, o1, do, l1, is_causal=causal, sinks=sinks)
    api.poll_status()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    for a, b in zip(g0, g1[:3]):
        assert torch.equal(a, b)
    assert torch.equal(g1[3], torch.zeros_like(sinks))


def test_sink_gradient_is_reproducible():
    shape = Shape(2, 8, 2, 300, 300, 128)
    q, k, v, do = (t.cuda() for t in draw(shape, 104, "bf16"))
    sinks = draw_sinks(shape.Hq, 105).cuda()
    o, lse = api.attention_forward(q, k, v, is_causal=True, sinks=sinks)
    runs = [api.attention_backward(q, k, v, o, do, lse, is_causal=True, sinks=sinks)[3].clone()
            for _ in range(3)]
    api.poll_status()
    assert all(torch.equal(runs[0], r) for r in runs[1:])


def test_sinks_with_blhd_views_match_the_oracle():
    shape = Shape(1, 8, 2, 180, 180, 64)
    q, k, v, do = draw(shape, 106, "bf16")
    sinks = draw_sinks(shape.Hq, 107)
    qs, ks, vs, dos = (t.transpose(1, 2).contiguous().cuda().transpose(1, 2) for t in (q, k, v, do))
    o, lse = api.attention_forward(qs, ks, vs, is_causal=True, sinks=sinks.cuda())
    dq, dk, dv, ds = api.attention_backward(qs, ks, vs, o, dos, lse, is_causal=True,
                                            sinks=sinks.cuda())
    api.poll_status()
    scale = 1.0 / math.sqrt(shape.D)
    qn, kn, vn, don = (as_f64(t) for t in (q, k, v, do))
    o_ref, lse_ref = oracle.sdpa_forward(qn, kn, vn, scale, True, sinks=as_f64(sinks))
    check_forward("bf16", as_f64(o), as_f64(lse), o_ref, lse_ref, "blhd sinks")
    refs = oracle.sdpa_backward(qn, kn, vn, don, scale, True, sinks=as_f64(sinks))
    for name, g, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs[:3]):
        check_grad("bf16", name, as_f64(g), ref, "blhd sinks")
    check_dsinks("bf16", as_f64(ds), refs[3], "blhd sinks")


def test_autograd_sinks_receive_gradients():
    shape = Shape(2, 8, 2, 128, 192, 128)
    q, k, v, do = draw(shape, 108, "bf16")
    sinks = draw_sinks(shape.Hq, 109)
    qd, kd, vd = (t.cuda().requires_grad_(True) for t in (q, k, v))
    sd = sinks.cuda().requires_grad_(True)
    out = autograd.scaled_dot_product_attention(qd, kd, vd, is_causal=True, enable_gqa=True,
                                                sinks=sd)
    out.backward(do.cuda())
    torch.cuda.synchronize()
    scale = 1.0 / math.sqrt(shape.D)
    qn, kn, vn, don = (as_f64(t) for t in (q, k, v, do))
    refs = oracle.sdpa_backward(qn, kn, vn, don, scale, True, sinks=as_f64(sinks))
    for name, leaf, ref in zip(("dq", "dk", "dv"), (qd, kd, vd), refs[:3]):
        check_grad("bf16", name, as_f64(leaf.grad), ref, "autograd sinks")
    check_dsinks("bf16", as_f64(sd.grad), refs[3], "autograd sinks")


def test_sinks_at_a_larger_size_on_sampled_rows():
    """Headline-like shape (GQA 4, D = 128, causal, 2048 rows): the oracle recomputes a
    few sampled query rows of several heads; the sink gradient is checked against its
    definition, −Σ exp(σ − lse)·(dO·O), evaluated in fp64 on the GPU's own O and lse
    (both checked on the samples)."""
    shape = Shape(1, 8, 2, 2048, 2048, 128)
    q, k, v, do = draw(shape, 110, "bf16")
    sinks = draw_sinks(shape.Hq, 111)
    scale = 1.0 / math.sqrt(shape.D)
    qd, kd, vd, dod, sd = (t.cuda() for t in (q, k, v, do, sinks))
    o, lse = api.attention_forward(qd, kd, vd, scale=scale, is_causal=True, sinks=sd)
    _, _, _, ds = api.attention_backward(qd, kd, vd, o, dod, lse, scale=scale, is_causal=True,
                                         sinks=sd)
    api.poll_status()
    rows = np.array([0, 1, 127, 128, 1000, 2047])
    G = shape.Hq // shape.Hkv
    for h in (0, 1, 2, 7):
        o_ref, lse_ref = oracle.head_forward(as_f64(q[0, h]), as_f64(k[0, h // G]),
                                             as_f64(v[0, h // G]), scale, True, rows=rows,
                                             sink=float(sinks[h]))
        check_forward("bf16", as_f64(o[0, h])[rows], as_f64(lse[0, h])[rows], o_ref, lse_ref,
                      f"h={h}")
    # dsink from the GPU's own O and lse (both checked above on samples), in fp64.
    on, ln, don = as_f64(o), as_f64(lse), as_f64(do)
    delta = (on * don).sum(-1)
    want = -(np.exp(as_f64(sinks)[None, :, None] - ln) * delta).sum(axis=(0, 2))
    check_dsinks("bf16", as_f64(ds), want, "sampled")
