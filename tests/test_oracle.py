"""Pins for the CPU oracle: checks against facts that do not come from the oracle itself.

Each test names the fact it uses: hand-derived closed forms (``tests/golden``), central
finite differences of the forward, special cases with closed forms, invariants of
softmax attention, and an independent library routine (PyTorch's CPU SDPA in float64,
as a second opinion only).  ``test_planted_mistakes_are_caught`` plants plausible bugs
in a copy of the oracle and checks that at least one pin fails for each.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import ref

HERE = os.path.dirname(os.path.abspath(__file__))


def rnd(rng, *shape):
    return rng.standard_normal(shape)


def make(rng, B=1, Hq=2, Hkv=1, Lq=5, Lkv=6, D=4):
    q = rnd(rng, B, Hq, Lq, D)
    k = rnd(rng, B, Hkv, Lkv, D)
    v = rnd(rng, B, Hkv, Lkv, D)
    do = rnd(rng, B, Hq, Lq, D)
    return q, k, v, do


# ----------------------------------------------------------------------------- golden
def _exact(x):
    """[num, den] -> num/den ; [num, den, c] -> num/den * ln(c); nested lists recurse."""
    if isinstance(x, list) and x and not isinstance(x[0], list):
        val = x[0] / x[1]
        return val * math.log(x[2]) if len(x) == 3 else val
    return [_exact(y) for y in x]


def _cases():
    with open(os.path.join(HERE, "golden", "closed_form_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_closed_form_fixtures(case):
    q = np.array(case["q"])
    k = np.array(_exact(case["k_exact"]))
    v = np.array(case["v"])
    do = np.array(case["dout"])
    assert np.allclose(k, np.array(case["k"]), atol=1e-15)
    kw = {}
    if "sinks_exact" in case:
        kw["sinks"] = np.array(_exact(case["sinks_exact"]))
    if "mask_bool" in case:
        kw["mask"] = np.array(case["mask_bool"], dtype=bool)
    if "mask_exact" in case:
        kw["mask"] = np.array(_exact(case["mask_exact"]))
    o, lse = oracle.sdpa_forward(q, k, v, case["scale"], case["is_causal"], **kw)
    grads = oracle.sdpa_backward(q, k, v, do, case["scale"], case["is_causal"], **kw)
    dq, dk, dv = grads[:3]
    if "dsinks" in case:
        np.testing.assert_allclose(grads[3], np.array(_exact(case["dsinks"])), atol=1e-13)
    np.testing.assert_allclose(o, np.array(_exact(case["o"])), atol=1e-13)
    np.testing.assert_allclose(lse, np.array(_exact(case["lse"])), atol=1e-13)
    np.testing.assert_allclose(dq, np.array(_exact(case["dq"])), atol=1e-13)
    np.testing.assert_allclose(dk, np.array(_exact(case["dk"])), atol=1e-13)
    np.testing.assert_allclose(dv, np.array(_exact(case["dv"])), atol=1e-13)


# ----------------------------------------------------------------- finite differences
def _loss(q, k, v, do, scale, causal, impl=None):
    impl = impl or oracle
    o, _ = impl.sdpa_forward(q, k, v, scale, causal)
    return float((o * do).sum())


def _fd_grad(x, f, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = x[i]
        x[i] = old + h
        fp = f()
        x[i] = old - h
        fm = f()
        x[i] = old
        g[i] = (fp - fm) / (2 * h)
    return g


FD_CASES = [
    dict(B=1, Hq=2, Hkv=1, Lq=5, Lkv=6, D=4, causal=False),
    dict(B=1, Hq=2, Hkv=1, Lq=5, Lkv=6, D=4, causal=True),
    dict(B=2, Hq=3, Hkv=3, Lq=4, Lkv=4, D=3, causal=True),
    dict(B=1, Hq=4, Hkv=2, Lq=7, Lkv=3, D=2, causal=True),
    dict(B=1, Hq=1, Hkv=1, Lq=1, Lkv=5, D=3, causal=False),
    dict(B=1, Hq=2, Hkv=1, Lq=4, Lkv=7, D=3, causal=2),      # bottom-right causal
]


@pytest.mark.parametrize("case", FD_CASES, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_backward_matches_finite_differences(case, impl=None):
    impl = impl or oracle
    rng = np.random.default_rng(11)
    c = dict(case)
    causal = c.pop("causal")
    q, k, v, do = make(rng, **c)
    scale = 0.7
    dq, dk, dv = impl.sdpa_backward(q, k, v, do, scale, causal)
    f = lambda: _loss(q, k, v, do, scale, causal, impl)  # noqa: E731
    np.testing.assert_allclose(dq, _fd_grad(q, f), atol=1e-7, rtol=1e-6)
    np.testing.assert_allclose(dk, _fd_grad(k, f), atol=1e-7, rtol=1e-6)
    np.testing.assert_allclose(dv, _fd_grad(v, f), atol=1e-7, rtol=1e-6)


# ----------------------------------------------------------------- special cases
def test_rows_of_p_sum_to_one(impl=None):
    """With V = identity (Lkv <= D), O is P itself: every row is a probability vector."""
    impl = impl or oracle
    rng = np.random.default_rng(1)
    for causal in (False, True):
        q = rnd(rng, 1, 2, 9, 8)
        k = rnd(rng, 1, 2, 8, 8)
        v = np.broadcast_to(np.eye(8), (1, 2, 8, 8)).copy()
        o, lse = impl.sdpa_forward(q, k, v, 0.9, causal)
        assert (o >= 0).all()
        np.testing.assert_allclose(o.sum(-1), 1.0, atol=1e-14)
        if causal:  # masked entries are exactly zero
            for i in range(8):
                assert (o[..., i, i + 1:] == 0).all()
        # lse is log of the row sum of exp(scores): check against P's definition
        s = np.einsum("bhid,bhjd->bhij", q, k) * 0.9
        j = np.arange(8)
        for i in range(9):
            vis = j <= i if causal else np.ones(8, bool)
            np.testing.assert_allclose(o[..., i, vis], np.exp(s[..., i, vis] - lse[..., i, None]),
                                       atol=1e-13)


def test_constant_v_gives_constant_output(impl=None):
    impl = impl or oracle
    rng = np.random.default_rng(2)
    q, k, _, _ = make(rng, B=2, Hq=4, Hkv=2, Lq=6, Lkv=9, D=5)
    c = rnd(rng, 5)
    v = np.broadcast_to(c, (2, 2, 9, 5)).copy()
    for causal in (False, True):
        o, _ = impl.sdpa_forward(q, k, v, 0.3, causal)
        np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), atol=1e-13)


def test_causal_first_row_attends_only_to_key0(impl=None):
    impl = impl or oracle
    rng = np.random.default_rng(3)
    q, k, v, do = make(rng, B=1, Hq=4, Hkv=2, Lq=6, Lkv=6, D=5)
    scale = 0.45
    o, lse = impl.sdpa_forward(q, k, v, scale, True)
    dq, _, _ = impl.sdpa_backward(q, k, v, do, scale, True)
    for h in range(4):
        g = h // 2
        np.testing.assert_allclose(o[0, h, 0], v[0, g, 0], atol=1e-14)
        np.testing.assert_allclose(lse[0, h, 0], scale * q[0, h, 0] @ k[0, g, 0], atol=1e-14)
        np.testing.assert_allclose(dq[0, h, 0], 0.0, atol=1e-14)


def test_single_key(impl=None):
    """Lkv = 1: O = v0, lse = scale q.k0, dQ = dK = 0, dV0 = sum of dO over the group."""
    impl = impl or oracle
    rng = np.random.default_rng(4)
    q, k, v, do = make(rng, B=2, Hq=6, Hkv=2, Lq=5, Lkv=1, D=3)
    for causal in (False, True):
        o, lse = impl.sdpa_forward(q, k, v, 1.3, causal)
        dq, dk, dv = impl.sdpa_backward(q, k, v, do, 1.3, causal)
        kk = np.repeat(k, 3, axis=1)
        np.testing.assert_allclose(o, np.repeat(v, 3, axis=1).repeat(5, axis=2), atol=1e-14)
        np.testing.assert_allclose(lse, 1.3 * np.einsum("bhid,bhjd->bhi", q, kk), atol=1e-13)
        np.testing.assert_allclose(dq, 0.0, atol=1e-13)
        np.testing.assert_allclose(dk, 0.0, atol=1e-13)
        np.testing.assert_allclose(dv[:, :, 0], do.reshape(2, 2, 3 * 5, 3).sum(2), atol=1e-13)


def test_zero_scale_is_uniform_attention(impl=None):
    """scale = 0: O is the mean of V (causal: the prefix mean); lse = log(#visible keys)."""
    impl = impl or oracle
    rng = np.random.default_rng(5)
    q, k, v, _ = make(rng, B=1, Hq=2, Hkv=1, Lq=7, Lkv=5, D=3)
    o, lse = impl.sdpa_forward(q, k, v, 0.0, False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(2, keepdims=True), o.shape), atol=1e-14)
    np.testing.assert_allclose(lse, math.log(5), atol=1e-14)
    o, lse = impl.sdpa_forward(q, k, v, 0.0, True)
    for i in range(7):
        n = min(i + 1, 5)
        np.testing.assert_allclose(o[0, :, i], np.broadcast_to(v[0, 0, :n].mean(0), (2, 3)),
                                   atol=1e-14)
        np.testing.assert_allclose(lse[0, :, i], math.log(n), atol=1e-14)


# ----------------------------------------------------------------- invariants
def test_gradient_sums(impl=None):
    """Rows of dS sum to 0, so dK sums to 0 over keys; dV sums to the sum of dO."""
    impl = impl or oracle
    rng = np.random.default_rng(6)
    q, k, v, do = make(rng, B=2, Hq=4, Hkv=2, Lq=8, Lkv=11, D=6)
    for causal in (False, True):
        dq, dk, dv = impl.sdpa_backward(q, k, v, do, 0.6, causal)
        np.testing.assert_allclose(dk.sum(2), 0.0, atol=1e-12)
        np.testing.assert_allclose(dv.sum(2), do.reshape(2, 2, 2 * 8, 6).sum(2), atol=1e-12)


def test_key_shift_invariance(impl=None):
    """K <- K + c: O and dQ unchanged (every score of row i shifts by scale q_i.c),
    lse shifts by scale q_i.c."""
    impl = impl or oracle
    rng = np.random.default_rng(7)
    q, k, v, do = make(rng, B=1, Hq=4, Hkv=2, Lq=6, Lkv=7, D=5)
    c = rnd(rng, 5)
    for causal in (False, True):
        o0, l0 = impl.sdpa_forward(q, k, v, 0.8, causal)
        o1, l1 = impl.sdpa_forward(q, k + c, v, 0.8, causal)
        dq0, dk0, dv0 = impl.sdpa_backward(q, k, v, do, 0.8, causal)
        dq1, dk1, dv1 = impl.sdpa_backward(q, k + c, v, do, 0.8, causal)
        np.testing.assert_allclose(o1, o0, atol=1e-12)
        np.testing.assert_allclose(l1 - l0, 0.8 * q @ c, atol=1e-12)
        np.testing.assert_allclose(dq1, dq0, atol=1e-12)
        np.testing.assert_allclose(dk1, dk0, atol=1e-12)
        np.testing.assert_allclose(dv1, dv0, atol=1e-12)


def test_gqa_equals_repeated_kv_heads(impl=None):
    """GQA = MHA on KV heads repeated G times in place (contiguous groups), with dK/dV
    summed over each group."""
    impl = impl or oracle
    rng = np.random.default_rng(8)
    q, k, v, do = make(rng, B=2, Hq=6, Hkv=2, Lq=5, Lkv=7, D=4)
    for causal in (False, True):
        o, lse = impl.sdpa_forward(q, k, v, 0.5, causal)
        dq, dk, dv = impl.sdpa_backward(q, k, v, do, 0.5, causal)
        kr, vr = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
        o2, lse2 = impl.sdpa_forward(q, kr, vr, 0.5, causal)
        dq2, dk2, dv2 = impl.sdpa_backward(q, kr, vr, do, 0.5, causal)
        np.testing.assert_allclose(o, o2, atol=1e-14)
        np.testing.assert_allclose(lse, lse2, atol=1e-14)
        np.testing.assert_allclose(dq, dq2, atol=1e-13)
        np.testing.assert_allclose(dk, dk2.reshape(2, 2, 3, 7, 4).sum(2), atol=1e-13)
        np.testing.assert_allclose(dv, dv2.reshape(2, 2, 3, 7, 4).sum(2), atol=1e-13)


def test_mha_equals_independent_heads(impl=None):
    """Hq = Hkv: every head is an independent attention problem."""
    impl = impl or oracle
    rng = np.random.default_rng(9)
    q, k, v, do = make(rng, B=2, Hq=3, Hkv=3, Lq=4, Lkv=6, D=3)
    o, lse = impl.sdpa_forward(q, k, v, 0.5, True)
    dq, dk, dv = impl.sdpa_backward(q, k, v, do, 0.5, True)
    for b in range(2):
        for h in range(3):
            oh, lh = impl.sdpa_forward(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1],
                                       v[b:b + 1, h:h + 1], 0.5, True)
            gh = impl.sdpa_backward(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1],
                                    v[b:b + 1, h:h + 1], do[b:b + 1, h:h + 1], 0.5, True)
            np.testing.assert_allclose(o[b, h], oh[0, 0], atol=1e-14)
            np.testing.assert_allclose(lse[b, h], lh[0, 0], atol=1e-14)
            for full, part in zip((dq, dk, dv), gh):
                np.testing.assert_allclose(full[b, h], part[0, 0], atol=1e-14)


def test_row_blocks_and_sampled_rows_agree():
    rng = np.random.default_rng(10)
    q, k, v, do = make(rng, B=1, Hq=4, Hkv=2, Lq=37, Lkv=29, D=4)
    for causal in (False, True):
        o, lse = oracle.sdpa_forward(q, k, v, 0.4, causal)
        o2, lse2 = oracle.sdpa_forward(q, k, v, 0.4, causal, row_block=8)
        g = oracle.sdpa_backward(q, k, v, do, 0.4, causal)
        g2 = oracle.sdpa_backward(q, k, v, do, 0.4, causal, row_block=5)
        np.testing.assert_allclose(o, o2, atol=1e-14)
        np.testing.assert_allclose(lse, lse2, atol=1e-14)
        for a, b in zip(g, g2):
            np.testing.assert_allclose(a, b, atol=1e-13)
        rows = np.array([36, 0, 17, 5])
        orow, lrow = oracle.head_forward(q[0, 3], k[0, 1], v[0, 1], 0.4, causal, rows=rows)
        np.testing.assert_allclose(orow, o[0, 3, rows], atol=1e-14)
        np.testing.assert_allclose(lrow, lse[0, 3, rows], atol=1e-14)


def test_float32_inputs_are_upcast_exactly():
    rng = np.random.default_rng(12)
    q, k, v, do = (x.astype(np.float32) for x in make(rng))
    o, _ = oracle.sdpa_forward(q, k, v, 0.5, False)
    o64, _ = oracle.sdpa_forward(q.astype(np.float64), k.astype(np.float64),
                                 v.astype(np.float64), 0.5, False)
    assert o.dtype == np.float64
    np.testing.assert_array_equal(o, o64)


# ----------------------------------------------------------------- library second opinion
def test_matches_torch_cpu_float64():
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    rng = np.random.default_rng(13)
    q, k, v, do = make(rng, B=2, Hq=4, Hkv=2, Lq=9, Lkv=9, D=8)
    for causal in (False, True):
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        kr = tk.repeat_interleave(2, dim=1)
        vr = tv.repeat_interleave(2, dim=1)
        o = F.scaled_dot_product_attention(tq, kr, vr, is_causal=causal, scale=0.35)
        o.backward(torch.tensor(do))
        oo, _ = oracle.sdpa_forward(q, k, v, 0.35, causal)
        dq, dk, dv = oracle.sdpa_backward(q, k, v, do, 0.35, causal)
        np.testing.assert_allclose(oo, o.detach().numpy(), atol=1e-12)
        np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
        np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
        np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)


def test_masks_match_torch_cpu_float64():
    """Second opinion for the mask reading: torch's CPU SDPA in float64 with the same
    boolean and additive attn_mask (no row fully hidden, where torch's conventions vary)."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    rng = np.random.default_rng(14)
    q, k, v, do = make(rng, B=2, Hq=4, Hkv=2, Lq=7, Lkv=9, D=8)
    boolean = rng.random((2, 1, 7, 9)) < 0.6
    boolean[..., 0] = True
    additive = rng.standard_normal((4, 7, 9))
    additive[rng.random(additive.shape) < 0.2] = -np.inf
    additive[..., 1] = 0.0
    for mask in (boolean, additive):
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        o = F.scaled_dot_product_attention(tq, tk.repeat_interleave(2, dim=1),
                                           tv.repeat_interleave(2, dim=1),
                                           attn_mask=torch.tensor(mask), scale=0.35)
        o.backward(torch.tensor(do))
        oo, _ = oracle.sdpa_forward(q, k, v, 0.35, False, mask=mask)
        dq, dk, dv = oracle.sdpa_backward(q, k, v, do, 0.35, False, mask=mask)
        np.testing.assert_allclose(oo, o.detach().numpy(), atol=1e-12)
        np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
        np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
        np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)


# ----------------------------------------------------------------- bottom-right causal
def test_bottom_right_equals_padded_top_left(impl=None):
    """The bottom-right mask (key j hidden from query i when j > i + Lkv - Lq) is the
    top-left mask of a problem with Lkv - Lq extra query rows in front: its rows are the
    last Lq rows of that problem, and with zero output gradient on the extra rows the
    gradients of K and V are the same."""
    impl = impl or oracle
    rng = np.random.default_rng(41)
    B, Hq, Hkv, Lq, Lkv, D = 1, 4, 2, 5, 9, 3
    q = rng.standard_normal((B, Hq, Lq, D))
    k = rng.standard_normal((B, Hkv, Lkv, D))
    v = rng.standard_normal((B, Hkv, Lkv, D))
    do = rng.standard_normal((B, Hq, Lq, D))
    pad = Lkv - Lq
    qf = np.concatenate([rng.standard_normal((B, Hq, pad, D)), q], axis=2)
    dof = np.concatenate([np.zeros((B, Hq, pad, D)), do], axis=2)
    o, lse = impl.sdpa_forward(q, k, v, 0.7, 2)
    of, lsef = impl.sdpa_forward(qf, k, v, 0.7, True)
    np.testing.assert_allclose(o, of[:, :, pad:], atol=1e-13)
    np.testing.assert_allclose(lse, lsef[:, :, pad:], atol=1e-13)
    dq, dk, dv = impl.sdpa_backward(q, k, v, do, 0.7, 2)
    dqf, dkf, dvf = impl.sdpa_backward(qf, k, v, dof, 0.7, True)
    np.testing.assert_allclose(dq, dqf[:, :, pad:], atol=1e-12)
    np.testing.assert_allclose(dk, dkf, atol=1e-12)
    np.testing.assert_allclose(dv, dvf, atol=1e-12)


def test_bottom_right_square_and_single_query(impl=None):
    """Lq = Lkv: bottom-right is top-left.  Lq = 1: the single query sees every key."""
    impl = impl or oracle
    rng = np.random.default_rng(42)
    q, k, v = (rng.standard_normal((1, 2, 6, 4)) for _ in range(3))
    for a, b in zip(impl.sdpa_forward(q, k, v, 0.5, 2), impl.sdpa_forward(q, k, v, 0.5, True)):
        np.testing.assert_allclose(a, b, atol=1e-14)
    q1 = q[:, :, :1]
    for a, b in zip(impl.sdpa_forward(q1, k, v, 0.5, 2), impl.sdpa_forward(q1, k, v, 0.5, False)):
        np.testing.assert_allclose(a, b, atol=1e-14)
    with pytest.raises(ValueError):
        impl.sdpa_forward(q, k[:, :, :3], v[:, :, :3], 0.5, 2)  # Lq > Lkv


# ----------------------------------------------------------------- attention sinks
def test_sink_at_minus_infinity_is_no_sink(impl=None):
    """exp(-inf) = 0: a sink of -inf leaves every output as without a sink and its own
    gradient is zero."""
    impl = impl or oracle
    rng = np.random.default_rng(51)
    q, k, v, do = make(rng, B=2, Hq=4, Hkv=2, Lq=5, Lkv=7, D=3)
    sinks = np.full(4, -np.inf)
    for causal in (False, True):
        for a, b in zip(impl.sdpa_forward(q, k, v, 0.6, causal, sinks=sinks),
                        impl.sdpa_forward(q, k, v, 0.6, causal)):
            np.testing.assert_allclose(a, b, atol=1e-14)
        r = impl.sdpa_backward(q, k, v, do, 0.6, causal, sinks=sinks)
        for a, b in zip(r[:3], impl.sdpa_backward(q, k, v, do, 0.6, causal)):
            np.testing.assert_allclose(a, b, atol=1e-14)
        np.testing.assert_array_equal(r[3], 0.0)


def test_sink_single_key_closed_form(impl=None):
    """One key with score s and a sink σ: O = v0 · e^s / (e^s + e^σ),
    lse = log(e^s + e^σ), and dσ = -Σ_i e^σ / (e^s_i + e^σ) · (dO_i · O_i)."""
    impl = impl or oracle
    rng = np.random.default_rng(52)
    q, k, v, do = make(rng, B=1, Hq=2, Hkv=1, Lq=3, Lkv=1, D=4)
    sinks = np.array([0.3, -1.2])
    o, lse = impl.sdpa_forward(q, k, v, 0.8, False, sinks=sinks)
    _, _, _, dsinks = impl.sdpa_backward(q, k, v, do, 0.8, False, sinks=sinks)
    for h in range(2):
        sc = 0.8 * q[0, h] @ k[0, 0, 0]
        w = 1.0 / (1.0 + np.exp(sinks[h] - sc))
        np.testing.assert_allclose(o[0, h], w[:, None] * v[0, 0, 0][None, :], atol=1e-14)
        np.testing.assert_allclose(lse[0, h], np.logaddexp(sc, sinks[h]), atol=1e-14)
        want = -np.sum((1.0 - w) * w * (do[0, h] @ v[0, 0, 0]))
        np.testing.assert_allclose(dsinks[h], want, atol=1e-13)


def test_sink_is_an_extra_key_with_zero_value(impl=None):
    """A sink σ behaves as one more key whose score is σ for every row and whose value is
    zero.  Build that key explicitly: append a coordinate 1 to every query and 0 to every
    key, and put a key (0, …, 0, σ/scale) with value 0 in front of the keys.  Without a
    mask, and with the bottom-right mask (which the extra front key leaves in place for
    the old keys and keeps visible to every row), the sink problem's outputs, logsumexp
    and gradients are those of the bigger problem, and dσ = dK_extra[D] / scale."""
    impl = impl or oracle
    rng = np.random.default_rng(53)
    B, Hq, Hkv, Lq, Lkv, D, scale = 2, 4, 2, 5, 7, 3, 0.7
    q, k, v, do = make(rng, B=B, Hq=Hq, Hkv=Hkv, Lq=Lq, Lkv=Lkv, D=D)
    sinks = np.array([0.4, -0.9, 1.3, 0.0])
    G = Hq // Hkv
    qa = np.concatenate([q, np.ones((B, Hq, Lq, 1))], axis=3)
    for causal in (False, 2):
        o, lse = impl.sdpa_forward(q, k, v, scale, causal, sinks=sinks)
        dq, dk, dv, dsinks = impl.sdpa_backward(q, k, v, do, scale, causal, sinks=sinks)
        for h in range(Hq):
            g = h // G
            ka = np.concatenate([k[:, g:g + 1], np.zeros((B, 1, Lkv, 1))], axis=3)
            extra = np.zeros((B, 1, 1, D + 1))
            extra[..., D] = sinks[h] / scale
            ka = np.concatenate([extra, ka], axis=2)
            va = np.concatenate([np.zeros((B, 1, 1, D)), v[:, g:g + 1]], axis=2)
            qh, doh = qa[:, h:h + 1], do[:, h:h + 1]
            oa, lsea = impl.sdpa_forward(qh, ka, va, scale, causal)
            np.testing.assert_allclose(o[:, h:h + 1], oa, atol=1e-13)
            np.testing.assert_allclose(lse[:, h:h + 1], lsea, atol=1e-13)
            dqa, dka, _ = impl.sdpa_backward(qh, ka, va, doh, scale, causal)
            np.testing.assert_allclose(dq[:, h:h + 1], dqa[..., :D], atol=1e-12)
            np.testing.assert_allclose(dsinks[h], dka[:, 0, 0, D].sum() / scale, atol=1e-12)
        # dK and dV of a KV head sum over its query heads; check them on the G = 1 view.
        for g in range(Hkv):
            hs = range(g * G, (g + 1) * G)
            dk_sum = np.zeros_like(k[:, g])
            dv_sum = np.zeros_like(v[:, g])
            for h in hs:
                ka = np.concatenate([k[:, g:g + 1], np.zeros((B, 1, Lkv, 1))], axis=3)
                extra = np.zeros((B, 1, 1, D + 1))
                extra[..., D] = sinks[h] / scale
                ka = np.concatenate([extra, ka], axis=2)
                va = np.concatenate([np.zeros((B, 1, 1, D)), v[:, g:g + 1]], axis=2)
                _, dka, dva = impl.sdpa_backward(qa[:, h:h + 1], ka, va, do[:, h:h + 1], scale,
                                                 causal)
                dk_sum += dka[:, 0, 1:, :D]
                dv_sum += dva[:, 0, 1:]
            np.testing.assert_allclose(dk[:, g], dk_sum, atol=1e-12)
            np.testing.assert_allclose(dv[:, g], dv_sum, atol=1e-12)


SINK_FD_CASES = [
    dict(B=2, Hq=2, Hkv=1, Lq=5, Lkv=6, D=4, causal=False),
    dict(B=1, Hq=4, Hkv=2, Lq=6, Lkv=4, D=3, causal=True),
    dict(B=1, Hq=2, Hkv=2, Lq=3, Lkv=6, D=2, causal=2),
]


@pytest.mark.parametrize("case", SINK_FD_CASES,
                         ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_sink_gradients_match_finite_differences(case, impl=None):
    impl = impl or oracle
    rng = np.random.default_rng(54)
    c = dict(case)
    causal = c.pop("causal")
    q, k, v, do = make(rng, **c)
    sinks = rng.standard_normal(c["Hq"])
    scale = 0.7

    def f():
        o, _ = impl.sdpa_forward(q, k, v, scale, causal, sinks=sinks)
        return float((o * do).sum())
    dq, dk, dv, dsinks = impl.sdpa_backward(q, k, v, do, scale, causal, sinks=sinks)
    np.testing.assert_allclose(dq, _fd_grad(q, f), atol=1e-7, rtol=1e-6)
    np.testing.assert_allclose(dk, _fd_grad(k, f), atol=1e-7, rtol=1e-6)
    np.testing.assert_allclose(dv, _fd_grad(v, f), atol=1e-7, rtol=1e-6)
    np.testing.assert_allclose(dsinks, _fd_grad(sinks, f), atol=1e-7, rtol=1e-6)


def _sink_fd_all(impl):
    for c in SINK_FD_CASES:
        test_sink_gradients_match_finite_differences(c, impl)


# ----------------------------------------------------------------- attention masks
def test_zero_and_all_true_masks_are_no_mask(impl=None):
    impl = impl or oracle
    rng = np.random.default_rng(61)
    q, k, v, do = make(rng, B=2, Hq=4, Hkv=2, Lq=5, Lkv=7, D=3)
    want_f = impl.sdpa_forward(q, k, v, 0.6, True)
    want_b = impl.sdpa_backward(q, k, v, do, 0.6, True)
    for mask in (np.zeros((5, 7)), np.ones((2, 4, 5, 7), dtype=bool)):
        for a, b in zip(impl.sdpa_forward(q, k, v, 0.6, True, mask=mask), want_f):
            np.testing.assert_allclose(a, b, atol=1e-14)
        for a, b in zip(impl.sdpa_backward(q, k, v, do, 0.6, True, mask=mask), want_b):
            np.testing.assert_allclose(a, b, atol=1e-14)


def test_lower_triangular_bool_mask_is_the_causal_flag(impl=None):
    """A boolean mask that keeps key j for query i iff j <= i + c is the causal mask with
    offset c (c = 0 top-left, Lkv - Lq bottom-right)."""
    impl = impl or oracle
    rng = np.random.default_rng(62)
    q, k, v, do = make(rng, B=1, Hq=2, Hkv=1, Lq=4, Lkv=7, D=3)
    for flag, c in ((True, 0), (2, 3)):
        mask = np.tril(np.ones((4, 7), dtype=bool), k=c)
        for a, b in zip(impl.sdpa_forward(q, k, v, 0.8, False, mask=mask),
                        impl.sdpa_forward(q, k, v, 0.8, flag)):
            np.testing.assert_allclose(a, b, atol=1e-14)
        for a, b in zip(impl.sdpa_backward(q, k, v, do, 0.8, False, mask=mask),
                        impl.sdpa_backward(q, k, v, do, 0.8, flag)):
            np.testing.assert_allclose(a, b, atol=1e-14)


def test_key_padding_mask_equals_truncated_keys(impl=None):
    """A [B, 1, 1, Lkv] boolean mask hiding keys n_b.. of batch b is the problem with K and V
    cut to their first n_b rows; the hidden keys get zero dK and dV."""
    impl = impl or oracle
    rng = np.random.default_rng(63)
    q, k, v, do = make(rng, B=2, Hq=4, Hkv=2, Lq=5, Lkv=8, D=3)
    ns = (3, 8)
    mask = np.zeros((2, 1, 1, 8), dtype=bool)
    for b, n in enumerate(ns):
        mask[b, :, :, :n] = True
    o, lse = impl.sdpa_forward(q, k, v, 0.7, False, mask=mask)
    dq, dk, dv = impl.sdpa_backward(q, k, v, do, 0.7, False, mask=mask)
    for b, n in enumerate(ns):
        sl = slice(b, b + 1)
        ot, lt = impl.sdpa_forward(q[sl], k[sl, :, :n], v[sl, :, :n], 0.7, False)
        np.testing.assert_allclose(o[sl], ot, atol=1e-13)
        np.testing.assert_allclose(lse[sl], lt, atol=1e-13)
        gq, gk, gv = impl.sdpa_backward(q[sl], k[sl, :, :n], v[sl, :, :n], do[sl], 0.7, False)
        np.testing.assert_allclose(dq[sl], gq, atol=1e-12)
        np.testing.assert_allclose(dk[sl, :, :n], gk, atol=1e-12)
        np.testing.assert_allclose(dv[sl, :, :n], gv, atol=1e-12)
        np.testing.assert_array_equal(dk[sl, :, n:], 0.0)
        np.testing.assert_array_equal(dv[sl, :, n:], 0.0)


def test_log_two_mask_equals_a_duplicated_key(impl=None):
    """Adding ln 2 to the score of key j gives it the weight of two copies of itself: the
    problem with key j (and its value) duplicated.  dQ is the same; key j's dK and dV are the
    sums over the two copies."""
    impl = impl or oracle
    rng = np.random.default_rng(64)
    q, k, v, do = make(rng, B=1, Hq=2, Hkv=1, Lq=5, Lkv=6, D=3)
    j = 2
    mask = np.zeros((5, 6))
    mask[:, j] = np.log(2.0)
    kd = np.concatenate([k, k[:, :, j:j + 1]], axis=2)
    vd = np.concatenate([v, v[:, :, j:j + 1]], axis=2)
    for a, b in zip(impl.sdpa_forward(q, k, v, 0.9, False, mask=mask),
                    impl.sdpa_forward(q, kd, vd, 0.9, False)):
        np.testing.assert_allclose(a, b, atol=1e-13)
    dq, dk, dv = impl.sdpa_backward(q, k, v, do, 0.9, False, mask=mask)
    gq, gk, gv = impl.sdpa_backward(q, kd, vd, do, 0.9, False)
    np.testing.assert_allclose(dq, gq, atol=1e-12)
    gk[:, :, j] += gk[:, :, 6]
    gv[:, :, j] += gv[:, :, 6]
    np.testing.assert_allclose(dk, gk[:, :, :6], atol=1e-12)
    np.testing.assert_allclose(dv, gv[:, :, :6], atol=1e-12)


def test_row_constant_mask_shifts_only_the_logsumexp(impl=None):
    """Softmax is invariant to a per-row constant: a mask c_i on every key of row i leaves O
    and every gradient unchanged and adds c_i to lse_i."""
    impl = impl or oracle
    rng = np.random.default_rng(65)
    q, k, v, do = make(rng, B=1, Hq=2, Hkv=1, Lq=5, Lkv=6, D=3)
    c = rng.standard_normal((1, 2, 5, 1)) * 3.0
    mask = np.broadcast_to(c, (1, 2, 5, 6))
    o, lse = impl.sdpa_forward(q, k, v, 0.9, True, mask=mask)
    o0, lse0 = impl.sdpa_forward(q, k, v, 0.9, True)
    np.testing.assert_allclose(o, o0, atol=1e-13)
    np.testing.assert_allclose(lse, lse0 + c[..., 0], atol=1e-13)
    for a, b in zip(impl.sdpa_backward(q, k, v, do, 0.9, True, mask=mask),
                    impl.sdpa_backward(q, k, v, do, 0.9, True)):
        np.testing.assert_allclose(a, b, atol=1e-12)


def test_per_query_head_masks_under_gqa(impl=None):
    """The mask is indexed by the query head: with GQA, each query head with its own mask
    equals that head run alone against its KV head."""
    impl = impl or oracle
    rng = np.random.default_rng(66)
    q, k, v, do = make(rng, B=1, Hq=4, Hkv=2, Lq=5, Lkv=6, D=3)
    mask = rng.standard_normal((1, 4, 5, 6))
    o, lse = impl.sdpa_forward(q, k, v, 0.8, False, mask=mask)
    dq, _, _ = impl.sdpa_backward(q, k, v, do, 0.8, False, mask=mask)
    for h in range(4):
        g = h // 2
        oh, lh = impl.sdpa_forward(q[:, h:h + 1], k[:, g:g + 1], v[:, g:g + 1], 0.8, False,
                                   mask=mask[:, h:h + 1])
        np.testing.assert_allclose(o[:, h:h + 1], oh, atol=1e-13)
        np.testing.assert_allclose(lse[:, h:h + 1], lh, atol=1e-13)
        gq, _, _ = impl.sdpa_backward(q[:, h:h + 1], k[:, g:g + 1], v[:, g:g + 1],
                                      do[:, h:h + 1], 0.8, False, mask=mask[:, h:h + 1])
        np.testing.assert_allclose(dq[:, h:h + 1], gq, atol=1e-12)


def test_fully_masked_row(impl=None):
    """A row that sees no key (reading: O = 0, lse = -inf, zero gradients) leaves the other
    rows, and dK and dV, as in the problem without that row; with a sink the sink alone
    fills the row: O = 0 and lse = the sink."""
    impl = impl or oracle
    rng = np.random.default_rng(67)
    q, k, v, do = make(rng, B=1, Hq=2, Hkv=1, Lq=5, Lkv=6, D=3)
    mask = np.ones((5, 6), dtype=bool)
    mask[3] = False
    keep = [0, 1, 2, 4]
    with np.errstate(all="raise"):
        o, lse = impl.sdpa_forward(q, k, v, 0.7, False, mask=mask)
        dq, dk, dv = impl.sdpa_backward(q, k, v, do, 0.7, False, mask=mask)
    np.testing.assert_array_equal(o[:, :, 3], 0.0)
    assert np.all(lse[:, :, 3] == -np.inf)
    np.testing.assert_array_equal(dq[:, :, 3], 0.0)
    o4, l4 = impl.sdpa_forward(q[:, :, keep], k, v, 0.7, False)
    np.testing.assert_allclose(o[:, :, keep], o4, atol=1e-13)
    np.testing.assert_allclose(lse[:, :, keep], l4, atol=1e-13)
    g4 = impl.sdpa_backward(q[:, :, keep], k, v, do[:, :, keep], 0.7, False)
    np.testing.assert_allclose(dq[:, :, keep], g4[0], atol=1e-12)
    np.testing.assert_allclose(dk, g4[1], atol=1e-12)
    np.testing.assert_allclose(dv, g4[2], atol=1e-12)
    sinks = np.array([0.5, -1.0])
    o, lse = impl.sdpa_forward(q, k, v, 0.7, False, mask=mask, sinks=sinks)
    np.testing.assert_array_equal(o[:, :, 3], 0.0)
    np.testing.assert_allclose(lse[0, :, 3], sinks, atol=1e-15)
    # A sink of -inf is no sink, also on the row that sees nothing: every output is the
    # no-sink one and the sink's gradient is exactly 0 (no 0/0 from the empty row).
    sinks = np.array([-np.inf, -np.inf])
    with np.errstate(all="raise"):
        o, lse = impl.sdpa_forward(q, k, v, 0.7, False, mask=mask, sinks=sinks)
        r = impl.sdpa_backward(q, k, v, do, 0.7, False, mask=mask, sinks=sinks)
    np.testing.assert_array_equal(o[:, :, 3], 0.0)
    assert np.all(lse[:, :, 3] == -np.inf)
    np.testing.assert_allclose(r[0], dq, atol=1e-14)
    np.testing.assert_allclose(r[1], dk, atol=1e-14)
    np.testing.assert_allclose(r[2], dv, atol=1e-14)
    np.testing.assert_array_equal(r[3], 0.0)


MASK_FD_CASES = [
    dict(B=1, Hq=2, Hkv=1, Lq=5, Lkv=6, D=3, causal=False),
    dict(B=2, Hq=4, Hkv=2, Lq=4, Lkv=7, D=2, causal=True),
    dict(B=1, Hq=2, Hkv=2, Lq=3, Lkv=6, D=3, causal=2),
]


@pytest.mark.parametrize("case", MASK_FD_CASES,
                         ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_masked_gradients_match_finite_differences(case, impl=None):
    """A random additive mask with some hidden keys (key 0 stays visible to every row)."""
    impl = impl or oracle
    rng = np.random.default_rng(68)
    c = dict(case)
    causal = c.pop("causal")
    q, k, v, do = make(rng, **c)
    mask = rng.standard_normal((c["B"], c["Hq"], c["Lq"], c["Lkv"]))
    mask[rng.random(mask.shape) < 0.3] = -np.inf
    mask[..., 0] = 0.0
    scale = 0.7

    def f():
        o, _ = impl.sdpa_forward(q, k, v, scale, causal, mask=mask)
        return float((o * do).sum())
    dq, dk, dv = impl.sdpa_backward(q, k, v, do, scale, causal, mask=mask)
    np.testing.assert_allclose(dq, _fd_grad(q, f), atol=1e-7, rtol=1e-6)
    np.testing.assert_allclose(dk, _fd_grad(k, f), atol=1e-7, rtol=1e-6)
    np.testing.assert_allclose(dv, _fd_grad(v, f), atol=1e-7, rtol=1e-6)


def _mask_fd_all(impl):
    for c in MASK_FD_CASES:
        test_masked_gradients_match_finite_differences(c, impl)


# ----------------------------------------------------------------- pins have teeth
PINS = [
    test_rows_of_p_sum_to_one,
    test_constant_v_gives_constant_output,
    test_causal_first_row_attends_only_to_key0,
    test_single_key,
    test_zero_scale_is_uniform_attention,
    test_gradient_sums,
    test_key_shift_invariance,
    test_gqa_equals_repeated_kv_heads,
    test_mha_equals_independent_heads,
    test_bottom_right_equals_padded_top_left,
    test_bottom_right_square_and_single_query,
    test_sink_at_minus_infinity_is_no_sink,
    test_sink_single_key_closed_form,
    test_sink_is_an_extra_key_with_zero_value,
    _sink_fd_all,
    test_zero_and_all_true_masks_are_no_mask,
    test_lower_triangular_bool_mask_is_the_causal_flag,
    test_key_padding_mask_equals_truncated_keys,
    test_log_two_mask_equals_a_duplicated_key,
    test_row_constant_mask_shifts_only_the_logsumexp,
    test_per_query_head_masks_under_gqa,
    test_fully_masked_row,
    _mask_fd_all,
]


def _mutant(name):
    """A copy of the oracle module with one plausible mistake planted (CPU only)."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("oracle_mutant_" + name, ref.__file__)
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    if name in ("causal_diag_masked", "causal_off_by_one"):
        shift = 0 if name == "causal_diag_masked" else 2

        def _scores(q_rows, k, scale, offset, row_idx, mask_rows=None):
            s = (q_rows @ k.T) * scale
            if mask_rows is not None:
                s = s + mask_rows
            if offset is not None:
                j = np.arange(k.shape[0])[None, :]
                s = np.where(j >= np.asarray(row_idx)[:, None] + offset + shift, -np.inf, s)
            return s
        m._scores = _scores
    elif name == "bottom_right_offset_off_by_one":
        orig = m._causal_offset

        def _causal_offset(is_causal, lq, lkv):
            off = orig(is_causal, lq, lkv)
            return off - 1 if is_causal == m.BOTTOM_RIGHT else off
        m._causal_offset = _causal_offset
    elif name == "lse_log2":
        orig = m._softmax_rows

        def _softmax_rows(s, sink=None):
            r = orig(s, sink)
            return (r[0], r[1] / math.log(2.0)) + tuple(r[2:])
        m._softmax_rows = _softmax_rows
    elif name == "gqa_modulo":
        def sdpa_forward(q, k, v, scale, is_causal, row_block=None, sinks=None, mask=None):
            B, Hq, Hkv, G = m._check(q, k, v)
            mask = m._full_mask(mask, q, k)
            o = np.empty(q.shape[:3] + (v.shape[3],))
            lse = np.empty(q.shape[:3])
            for b in range(B):
                for h in range(Hq):
                    g = h % Hkv
                    o[b, h], lse[b, h] = m.head_forward(
                        q[b, h], k[b, g], v[b, g], scale, is_causal,
                        sink=None if sinks is None else float(sinks[h]),
                        mask=None if mask is None else mask[b, h])
            return o, lse
        m.sdpa_forward = sdpa_forward
    elif name == "no_scale_in_dq":
        orig = m.head_backward

        def head_backward(q, k, v, dout, scale, is_causal, row_block=None, sink=None, mask=None):
            r = orig(q, k, v, dout, scale, is_causal, row_block, sink, mask)
            return ((r[0] / scale if scale else r[0]),) + tuple(r[1:])
        m.head_backward = head_backward
    elif name == "delta_dropped":
        def head_backward(q, k, v, dout, scale, is_causal, row_block=None, sink=None, mask=None):
            q, k, v, dout = (np.asarray(x, float) for x in (q, k, v, dout))
            off = m._causal_offset(is_causal, q.shape[0], k.shape[0])
            mv = None if mask is None else np.broadcast_to(m._mask_values(mask), (q.shape[0], k.shape[0]))
            sm = m._softmax_rows(m._scores(q, k, scale, off, np.arange(q.shape[0]), mv), sink)
            p = sm[0]
            ds = p * (dout @ v.T)
            r = (scale * ds @ k, scale * ds.T @ q, p.T @ dout)
            return r if sink is None else r + (0.0,)
        m.head_backward = head_backward
    elif name == "dk_transposed_operand":
        orig = m.head_backward

        def head_backward(q, k, v, dout, scale, is_causal, row_block=None, sink=None, mask=None):
            r = orig(q, k, v, dout, scale, is_causal, row_block, sink, mask)
            return (r[0], r[1][::-1].copy()) + tuple(r[2:])
        m.head_backward = head_backward
    elif name == "sink_missing_from_lse":
        orig = m._softmax_rows

        def _softmax_rows(s, sink=None):
            r = orig(s, sink)
            return (r[0], orig(s)[1]) + tuple(r[2:])
        m._softmax_rows = _softmax_rows
    elif name == "sink_gradient_sign":
        orig = m.head_backward

        def head_backward(q, k, v, dout, scale, is_causal, row_block=None, sink=None, mask=None):
            r = orig(q, k, v, dout, scale, is_causal, row_block, sink, mask)
            return r if sink is None else r[:3] + (-r[3],)
        m.head_backward = head_backward
    elif name == "sink_given_a_value":
        orig = m.head_forward

        def head_forward(q, k, v, scale, is_causal, rows=None, row_block=None, sink=None, mask=None):
            o, lse = orig(q, k, v, scale, is_causal, rows, row_block, sink, mask)
            if sink is not None:
                o = o + np.exp(sink - lse)[:, None] * np.asarray(v, float)[0][None, :]
            return o, lse
        m.head_forward = head_forward
    elif name == "mask_scaled":
        def _scores(q_rows, k, scale, offset, row_idx, mask_rows=None):
            s = q_rows @ k.T
            if mask_rows is not None:
                s = s + mask_rows
            s = s * scale
            if offset is not None:
                j = np.arange(k.shape[0])[None, :]
                s = np.where(j > np.asarray(row_idx)[:, None] + offset, -np.inf, s)
            return s
        m._scores = _scores
    elif name == "bool_mask_inverted":
        def _mask_values(mask):
            mask = np.asarray(mask)
            if mask.dtype == np.bool_:
                return np.where(mask, -np.inf, 0.0)
            return mask.astype(np.float64)
        m._mask_values = _mask_values
    elif name == "mask_by_kv_head":
        def sdpa_forward(q, k, v, scale, is_causal, row_block=None, sinks=None, mask=None):
            B, Hq, Hkv, G = m._check(q, k, v)
            mask = m._full_mask(mask, q, k)
            o = np.empty(q.shape[:3] + (v.shape[3],))
            lse = np.empty(q.shape[:3])
            for b in range(B):
                for h in range(Hq):
                    g = h // G
                    o[b, h], lse[b, h] = m.head_forward(
                        q[b, h], k[b, g], v[b, g], scale, is_causal,
                        sink=None if sinks is None else float(sinks[h]),
                        mask=None if mask is None else mask[b, g])
            return o, lse
        m.sdpa_forward = sdpa_forward
    elif name == "masked_row_nan":
        def _softmax_rows(s, sink=None):
            mx = s.max(axis=1, keepdims=True)
            if sink is not None:
                mx = np.maximum(mx, sink)
            e = np.exp(s - mx)
            l = e.sum(axis=1, keepdims=True)
            if sink is not None:
                es = np.exp(sink - mx)
                l = l + es
            p = e / l
            lse = (mx + np.log(l))[:, 0]
            return (p, lse, (es / l)[:, 0]) if sink is not None else (p, lse)
        m._softmax_rows = _softmax_rows
    elif name == "empty_row_sink_share_nan":
        # the sink's share of a row with no finite entry left as 0/0
        def _softmax_rows(s, sink=None):
            mx = s.max(axis=1, keepdims=True)
            if sink is not None:
                mx = np.maximum(mx, sink)
            mx = np.where(np.isfinite(mx), mx, 0.0)
            e = np.exp(s - mx)
            l = e.sum(axis=1, keepdims=True)
            if sink is not None:
                es = np.exp(sink - mx)
                l = l + es
            with np.errstate(divide="ignore", invalid="ignore"):
                p = np.where(l > 0, e / l, 0.0)
                lse = (mx + np.log(l))[:, 0]
                share = (es / l)[:, 0] if sink is not None else None
            return (p, lse, share) if sink is not None else (p, lse)
        m._softmax_rows = _softmax_rows
    elif name == "mask_as_large_finite_negative":
        # hiding keys with -1e9 instead of -inf: a row that sees no key becomes uniform
        orig = m._mask_values

        def _mask_values(mask):
            return np.maximum(orig(mask), -1e9)
        m._mask_values = _mask_values
    elif name == "mask_subtracted":
        def _scores(q_rows, k, scale, offset, row_idx, mask_rows=None):
            s = (q_rows @ k.T) * scale
            if mask_rows is not None:
                s = s - np.where(np.isneginf(mask_rows), np.inf, mask_rows)
            if offset is not None:
                j = np.arange(k.shape[0])[None, :]
                s = np.where(j > np.asarray(row_idx)[:, None] + offset, -np.inf, s)
            return s
        m._scores = _scores
    elif name == "sink_gradient_without_delta":
        orig = m.head_backward

        def head_backward(q, k, v, dout, scale, is_causal, row_block=None, sink=None, mask=None):
            r = orig(q, k, v, dout, scale, is_causal, row_block, sink, mask)
            if sink is None:
                return r
            q64, k64 = np.asarray(q, float), np.asarray(k, float)
            off = m._causal_offset(is_causal, q64.shape[0], k64.shape[0])
            mv = None if mask is None else np.broadcast_to(m._mask_values(mask), (q64.shape[0], k64.shape[0]))
            sm = m._softmax_rows(m._scores(q64, k64, scale, off, np.arange(q64.shape[0]), mv), sink)
            return r[:3] + (-float(sm[2].sum()),)
        m.head_backward = head_backward
    else:
        raise KeyError(name)
    return m


@pytest.mark.parametrize("name", ["causal_diag_masked", "causal_off_by_one", "lse_log2", "gqa_modulo",
                                  "no_scale_in_dq", "delta_dropped", "dk_transposed_operand",
                                  "bottom_right_offset_off_by_one", "sink_missing_from_lse",
                                  "sink_gradient_sign", "sink_given_a_value", "mask_scaled",
                                  "bool_mask_inverted", "mask_by_kv_head", "masked_row_nan",
                                  "mask_as_large_finite_negative", "mask_subtracted", "empty_row_sink_share_nan",
                                  "sink_gradient_without_delta"])
def test_planted_mistakes_are_caught(name):
    mutant = _mutant(name)
    failures = 0
    checks = PINS + [lambda impl: [test_backward_matches_finite_differences(c, impl)
                                   for c in FD_CASES]]
    with np.errstate(all="ignore"):
        for pin in checks:
            try:
                pin(impl=mutant)
            except (AssertionError, FloatingPointError, ValueError):
                failures += 1
    assert failures > 0, f"no pin caught the planted mistake {name!r}"
