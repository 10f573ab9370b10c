"""Strided layouts: the same computation with every tensor stored as [B, L, H, D] (rows of
all heads together, seen as [B, H, L, D] through .transpose(1, 2)), or as views into one
fused [B, L, 3, H, D] projection output, passed to the library with their strides.

Each kernel family must give results bit-identical to the contiguous call (the arithmetic
is the same, only the addressing differs), and the autograd drop-in must take such views
without copying them."""
import math

import numpy as np
import pytest
import torch

import oracle
from parity_util import O_TOL, check_grad
from scaled_dot_product_flash_gb300 import _lib, api, autograd
from scaled_dot_product_flash_gb300.inputs import Shape, as_f64, draw

pytestmark = pytest.mark.gpu


def blhd(t):
    """[B, H, L, D] values stored as [B, L, H, D] on the GPU, returned as a [B, H, L, D] view."""
    return t.transpose(1, 2).contiguous().cuda().transpose(1, 2)


def empty_blhd(like):
    B, H, L, D = like.shape
    return torch.empty(B, L, H, D, device="cuda", dtype=like.dtype).transpose(1, 2)


CASES = [
    (Shape(2, 8, 2, 200, 200, 128), "bf16", True, _lib.PATH_AUTO),     # tensor cores, GQA, tail
    (Shape(1, 4, 4, 96, 160, 64), "f16", False, _lib.PATH_AUTO),       # tensor cores, Lq != Lkv
    (Shape(2, 8, 2, 4, 300, 128), "bf16", True, _lib.PATH_AUTO),       # short query, warp MMA
    (Shape(1, 4, 2, 40, 70, 32), "f32", True, _lib.PATH_AUTO),         # CUDA cores
    (Shape(1, 2, 2, 5, 90, 96), "f32", False, _lib.PATH_AUTO),         # short query, CUDA cores
    (Shape(1, 4, 2, 130, 130, 64), "bf16", True, _lib.PATH_SIMT),      # forced CUDA cores, bf16
    (Shape(1, 4, 2, 200, 330, 96), "bf16", True, _lib.PATH_AUTO),      # tensor cores, D = 96
    (Shape(1, 4, 2, 150, 200, 256), "bf16", True, _lib.PATH_AUTO),     # tensor cores, D = 256
    (Shape(2, 4, 4, 70, 130, 256), "f16", False, _lib.PATH_AUTO),      # D = 256, MHA
]


@pytest.mark.parametrize("shape,dtype,causal,path", CASES)
def test_blhd_matches_contiguous_bitwise(shape, dtype, causal, path):
    q, k, v, do = draw(shape, 91, dtype)
    with api.force_path(path):
        qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
        o_ref, lse_ref = api.attention_forward(qc, kc, vc, is_causal=causal)
        g_ref = api.attention_backward(qc, kc, vc, o_ref, doc, lse_ref, is_causal=causal)

        qs, ks, vs, dos = (blhd(t) for t in (q, k, v, do))
        assert not qs.is_contiguous()
        out = empty_blhd(qs)
        o, lse = api.attention_forward(qs, ks, vs, is_causal=causal, out=out)
        dq, dk, dv = empty_blhd(qs), empty_blhd(ks), empty_blhd(vs)
        api.attention_backward(qs, ks, vs, o, dos, lse, is_causal=causal, dq=dq, dk=dk, dv=dv)
        api.poll_status()
    assert torch.equal(o, o_ref)
    assert torch.equal(lse, lse_ref)
    for got, want in zip((dq, dk, dv), g_ref):
        assert torch.equal(got, want)


def test_fused_qkv_views_match_the_oracle():
    B, L, H, D = 2, 150, 4, 64
    rng = np.random.default_rng(92)
    qkv = torch.from_numpy(rng.standard_normal((B, L, 3, H, D), dtype=np.float32)).to(torch.bfloat16)
    do = torch.from_numpy(rng.standard_normal((B, H, L, D), dtype=np.float32)).to(torch.bfloat16)
    qkv_d = qkv.cuda()
    q, k, v = (qkv_d[:, :, n].transpose(1, 2) for n in range(3))  # views, no copies
    assert q.data_ptr() == qkv_d.data_ptr()
    o, lse = api.attention_forward(q, k, v, is_causal=True)
    dq, dk, dv = api.attention_backward(q, k, v, o, do.cuda(), lse, is_causal=True)
    api.poll_status()
    scale = 1.0 / math.sqrt(D)
    qn, kn, vn = (as_f64(qkv[:, :, n].transpose(1, 2)) for n in range(3))
    o_ref, _ = oracle.sdpa_forward(qn, kn, vn, scale, True)
    assert float(np.abs(as_f64(o) - o_ref).max()) <= O_TOL["bf16"]
    refs = oracle.sdpa_backward(qn, kn, vn, as_f64(do), scale, True)
    for name, g, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        check_grad("bf16", name, as_f64(g), ref, "fused qkv")


def test_autograd_takes_blhd_views_without_copies():
    shape = Shape(1, 8, 2, 96, 96, 128)
    q, k, v, do = draw(shape, 93, "bf16")
    leaves = [t.transpose(1, 2).contiguous().cuda().requires_grad_(True) for t in (q, k, v)]
    qv, kv, vv = (t.transpose(1, 2) for t in leaves)
    out = autograd.scaled_dot_product_attention(qv, kv, vv, is_causal=True, enable_gqa=True)
    assert out.stride() == qv.stride()  # the output keeps the input layout
    out.backward(do.cuda())
    torch.cuda.synchronize()
    scale = 1.0 / math.sqrt(shape.D)
    refs = oracle.sdpa_backward(as_f64(q), as_f64(k), as_f64(v), as_f64(do), scale, True)
    for name, leaf, ref in zip(("dq", "dk", "dv"), leaves, refs):
        check_grad("bf16", name, as_f64(leaf.grad.transpose(1, 2)), ref, "autograd blhd")
