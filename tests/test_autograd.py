"""The autograd wrapper and the ``scaled_dot_product_attention`` drop-in.

CPU tests check the argument handling that happens before anything reaches the library.
GPU tests run a forward and ``.backward()`` through torch autograd and compare the result
and the gradients with the CPU oracle, at the same tolerances as the parity tests, and
check that the drop-in agrees with ``torch.nn.functional.scaled_dot_product_attention``'s
conventions (top-left causal mask, default scale 1/sqrt(D), GQA by contiguous groups)."""
import math

import numpy as np
import pytest
import torch

import oracle
from parity_util import O_TOL, check_grad
from scaled_dot_product_flash_gb300 import autograd as sa
from scaled_dot_product_flash_gb300.inputs import Shape, as_f64, draw


def _cpu(shape=(1, 2, 8, 32)):
    return torch.zeros(shape)


def test_rejects_mask_gradients_and_dropout():
    q = k = v = _cpu()
    with pytest.raises(NotImplementedError):
        sa.scaled_dot_product_attention(q, k, v, attn_mask=torch.zeros(8, 8, requires_grad=True))
    with pytest.raises(ValueError):
        sa.scaled_dot_product_attention(q, k, v, attn_mask=torch.ones(8, 8, dtype=torch.bool),
                                        is_causal=True)
    with pytest.raises(NotImplementedError):
        sa.scaled_dot_product_attention(q, k, v, dropout_p=0.1)
    with pytest.raises(NotImplementedError):
        sa.scaled_dot_product_attention(torch.zeros(2, 8, 32), k, v)


def test_rejects_gqa_without_flag_and_bad_groups():
    q, kv = _cpu((1, 4, 8, 32)), _cpu((1, 2, 8, 32))
    with pytest.raises(ValueError):
        sa.scaled_dot_product_attention(q, kv, kv)
    with pytest.raises(ValueError):
        sa.scaled_dot_product_attention(_cpu((1, 3, 8, 32)), kv, kv, enable_gqa=True)
    with pytest.raises(ValueError):
        sa.scaled_dot_product_attention(q, kv, _cpu((1, 2, 9, 32)), enable_gqa=True)
    with pytest.raises(ValueError):
        sa.scaled_dot_product_attention(q, kv, kv, enable_gqa=True, scale=float("inf"))


def test_rejects_malformed_sinks():
    q = k = v = _cpu()
    with pytest.raises(ValueError):
        sa.scaled_dot_product_attention(q, k, v, sinks=torch.zeros(3))        # not Hq values
    with pytest.raises(ValueError):
        sa.scaled_dot_product_attention(q, k, v, sinks=torch.zeros(2, 1))     # not 1-D


@pytest.mark.gpu
@pytest.mark.parametrize("shape,dtype,causal", [
    (Shape(2, 8, 2, 200, 200, 128), "bf16", True),    # tensor-core path, GQA, ragged tail
    (Shape(1, 4, 4, 96, 160, 64), "f16", False),      # tensor-core path, Lq != Lkv
    (Shape(1, 4, 2, 40, 70, 32), "f32", True),        # CUDA-core path
    (Shape(2, 8, 2, 4, 300, 128), "bf16", False),     # short-query path
])
def test_autograd_matches_oracle(shape, dtype, causal):
    q, k, v, do = draw(shape, 77, dtype)
    qd, kd, vd = (t.cuda().requires_grad_(True) for t in (q, k, v))
    out = sa.scaled_dot_product_attention(qd, kd, vd, is_causal=causal,
                                          enable_gqa=shape.Hq != shape.Hkv)
    out.backward(do.cuda())
    torch.cuda.synchronize()
    scale = 1.0 / math.sqrt(shape.D)
    qn, kn, vn, don = (as_f64(t) for t in (q, k, v, do))
    o_ref, _ = oracle.sdpa_forward(qn, kn, vn, scale, causal)
    dq_ref, dk_ref, dv_ref = oracle.sdpa_backward(qn, kn, vn, don, scale, causal)
    err_o = float(np.max(np.abs(as_f64(out.detach()) - o_ref)))
    assert err_o <= O_TOL[dtype], f"O max-abs {err_o:.3e}"
    for name, g, ref in (("dq", qd.grad, dq_ref), ("dk", kd.grad, dk_ref), ("dv", vd.grad, dv_ref)):
        check_grad(dtype, name, as_f64(g), ref, "autograd")


@pytest.mark.gpu
def test_forward_only_skips_logsumexp_and_matches_torch_conventions():
    shape = Shape(1, 4, 2, 64, 80, 64)
    q, k, v, _ = (t.cuda() for t in draw(shape, 78, "f32"))
    with torch.no_grad():
        out = sa.scaled_dot_product_attention(q, k, v, is_causal=True, enable_gqa=True)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.double().cpu(), k.double().cpu().repeat_interleave(2, dim=1),
        v.double().cpu().repeat_interleave(2, dim=1), is_causal=True)
    assert float((out.double().cpu() - ref).abs().max()) < 1e-5
