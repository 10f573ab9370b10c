"""Plain fp64 CPU oracle for scaled-dot-product attention, forward and backward.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py``; never by the CUDA library or its binding.

Sources (web pages, cited by title and section):

* [PyTensor-SDPA] "PERF: detect scaled-dot-product-attention pattern and lower to
  mx.fast.scaled_dot_product_attention" (pymc-devs/pytensor issue 2090), section
  "Proposed change": the NumPy ``perform`` sketch computes scores = (Q Kᵀ)·scale,
  subtracts the row maximum, exponentiates, divides by the row sum and multiplies by V.
  The forward here is that definition, with the causal mask and grouped KV heads added.
* [MPS-SDPA] "MPS scaled_dot_product_attention (SDPA)" (PyTorch issue, stepcodex
  mirror), section "Problem - Unused second output tensor": the forward's second
  output (the per-row logsumexp) is what the backward needs.
* [MLX-VJP] "[Metal] Add Flash Attention VJP for training" (ml-explore/mlx PR 2995),
  sections "Implementation Notes" and "Key Features": logsumexp cached by the forward,
  GQA (several query heads share one KV head), causal masking; and the maintainer
  comment listing the backward's steps (recompute scores, load logsumexp,
  P = exp(S - LSE), gradients).
* [mps-flash-sdpa] "mps-flash-sdpa 0.1.0" (PyPI), section "Quick Start": the
  ``is_causal`` flag of ``F.scaled_dot_product_attention``.

Readings of points the pages leave open (each also listed in the design notes):

* logsumexp is the natural log of the row sum of exp(scale·q·k) over visible keys,
  including the scale; stored in fp32 by the GPU, fp64 here.
* causal is top-left aligned: key j is masked for query i when j > i, for any Lq, Lkv.
  Key 0 is always visible, so no row is ever fully masked.  ``is_causal = 2`` selects the
  bottom-right alignment instead (the last query sees every key): key j is masked for
  query i when j > i + (Lkv - Lq); it is defined for Lq <= Lkv only, where again key 0
  is always visible.
* GQA groups are contiguous: query head h reads KV head h // (Hq // Hkv).
* The backward is the textbook vector-Jacobian product of the forward with
  delta = rowsum(dO * O) taken from this oracle's own fp64 O.
* Attention sinks (optional, one logit per query head): the sink joins every row's
  softmax as one more entry with score ``sink[h]`` (natural-log units, like scale·q·k)
  and a zero value vector, so it enlarges the row sum and the logsumexp but adds nothing
  to O.  The backward is the same chain rule; the sink's own gradient is
  -sum_i p_sink,i · delta_i (its dP entry is zero because its value is zero).
* Attention masks (optional): an array broadcastable to [B, Hq, Lq, Lkv], indexed by the
  query head.  A boolean mask keeps key j for query i where it is True (the convention of
  ``F.scaled_dot_product_attention``'s ``attn_mask``); a float mask is added to
  scale·q·k before the softmax (−inf hides the key).  It combines with the causal mask.
  A row that sees no key at all (possible only with such a mask) has O = 0,
  lse = −inf and zero gradients (with a sink, the sink alone fills the row's softmax).
* The oracle does not clamp exponent arguments (the clamp mentioned in [MLX-VJP]
  "Implementation Notes" only guards the GPU's exp2 against overflow; after the row
  maximum is subtracted every argument is <= 0 already).

Arrays are NumPy, layout [B, H, L, D].  Inputs may be any float dtype; they are upcast
exactly to float64 (bf16/fp16 values are exactly representable).  Work goes one
(batch, head) at a time, and in blocks of whole query rows when ``row_block`` is given
so that long sequences fit in memory; every row is still computed over all its keys at
once, exactly as the definition says.

Parity: every function here is pinned by ``tests/test_oracle.py`` (finite differences,
closed forms, invariants, a hand-derived fixture under ``tests/golden/`` and a library
cross-check), so none is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "head_forward",
    "head_backward",
    "group_backward",
    "sdpa_forward",
    "sdpa_backward",
]


def _f64(x):
    return np.asarray(x, dtype=np.float64)


BOTTOM_RIGHT = 2


def _causal_offset(is_causal, lq, lkv):
    """None without a mask; otherwise the c for which key j is hidden from query i when
    j > i + c: 0 for the top-left mask, Lkv - Lq for the bottom-right one."""
    if not is_causal:
        return None
    if is_causal == BOTTOM_RIGHT:
        if lq > lkv:
            raise ValueError("the bottom-right causal mask needs Lq <= Lkv")
        return lkv - lq
    return 0


def _mask_values(mask):
    """A mask as additive fp64 values: boolean True -> 0, False -> -inf; floats as they are."""
    mask = np.asarray(mask)
    if mask.dtype == np.bool_:
        return np.where(mask, 0.0, -np.inf)
    return mask.astype(np.float64)


def _scores(q_rows, k, scale, offset, row_idx, mask_rows=None):
    """Scores of a block of query rows against all keys, masked.

    [PyTensor-SDPA] "Proposed change": scores = (q @ kᵀ) * scale.  ``mask_rows`` (the
    additive mask of these rows, or None) is added.  Causal ([mps-flash-sdpa] "Quick
    Start" ``is_causal``): the score of key j for absolute query row i = row_idx[r] is
    -inf when j > i + offset (offset None: no causal mask).
    """
    s = (q_rows @ k.T) * scale
    if mask_rows is not None:
        s = s + mask_rows
    if offset is not None:
        j = np.arange(k.shape[0])[None, :]
        s = np.where(j > np.asarray(row_idx)[:, None] + offset, -np.inf, s)
    return s


def _softmax_rows(s, sink=None):
    """Row softmax as [PyTensor-SDPA] "Proposed change" writes it, plus the logsumexp.

    Subtract the row maximum, exponentiate, divide by the row sum.  The logsumexp of
    the row ([MPS-SDPA] "Problem - Unused second output tensor") is max + log(sum).
    With a sink logit, the row is the scores plus one more entry equal to the sink; the
    returned P leaves that entry out, and p_sink (one per row) is returned as well.
    A row with no finite entry (every key hidden, no sink) gets P = 0 and lse = -inf.
    """
    m = s.max(axis=1, keepdims=True)
    if sink is not None:
        m = np.maximum(m, sink)
    m = np.where(np.isfinite(m), m, 0.0)  # rows with nothing visible: any finite shift
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    if sink is not None:
        es = np.exp(sink - m)
        l = l + es
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(l > 0, e / l, 0.0)
        lse = (m + np.log(l))[:, 0]
        if sink is not None:
            # A sink of -inf is no sink: with every key hidden too, the row is empty and
            # the sink's share is 0 like every other entry's.
            p_sink = np.where(l > 0, es / l, 0.0)[:, 0]
    if sink is not None:
        return p, lse, p_sink
    return p, lse


def _blocks(n, row_block):
    step = n if not row_block else int(row_block)
    for r0 in range(0, n, step):
        yield r0, min(n, r0 + step)


def head_forward(q, k, v, scale, is_causal, rows=None, row_block=None, sink=None, mask=None):
    """Forward of one head: O = softmax(scale·q kᵀ [+ masks]) v and its logsumexp.

    q: [Lq, D], k, v: [Lkv, D].  ``rows`` (optional, sorted or not) selects which query
    rows to compute; by default all.  ``sink``: this head's sink logit, or None.
    ``mask``: this head's [Lq, Lkv] mask (boolean or additive), or None.
    Returns (O [n, D], lse [n]) in float64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    if mask is not None:
        mask = np.broadcast_to(_mask_values(mask), (q.shape[0], k.shape[0]))
    off = _causal_offset(is_causal, q.shape[0], k.shape[0])
    idx = np.arange(q.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    o = np.empty((idx.size, v.shape[1]))
    lse = np.empty(idx.size)
    for a, b in _blocks(idx.size, row_block):
        sel = idx[a:b]
        mrows = None if mask is None else mask[sel]
        p, lse[a:b] = _softmax_rows(_scores(q[sel], k, scale, off, sel, mrows), sink)[:2]
        o[a:b] = p @ v
    return o, lse


def head_backward(q, k, v, dout, scale, is_causal, row_block=None, sink=None, mask=None):
    """Backward of one head (textbook VJP).  Returns (dq, dk_part, dv_part) in float64.

    Steps, per [MLX-VJP]'s description (recompute S, P = exp(S - LSE), then gradients)
    written as the plain chain rule of the forward:
        P   = softmax(S)                         (recomputed from q, k)
        O   = P v
        dV  = Pᵀ dO
        dP  = dO vᵀ
        δ   = rowsum(dO ∘ O)
        dS  = P ∘ (dP − δ)
        dQ  = scale · dS k
        dK  = scale · dSᵀ q
    dk_part and dv_part are this head's contribution to its KV head; the caller sums
    them over the query heads of the group.  With a sink logit, a fourth value is
    returned: the sink's gradient, -sum_i p_sink,i · δ_i.  ``mask``: as in head_forward.
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    if mask is not None:
        mask = np.broadcast_to(_mask_values(mask), (q.shape[0], k.shape[0]))
    off = _causal_offset(is_causal, q.shape[0], k.shape[0])
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dsink = 0.0
    for a, b in _blocks(q.shape[0], row_block):
        mrows = None if mask is None else mask[a:b]
        sm = _softmax_rows(_scores(q[a:b], k, scale, off, np.arange(a, b), mrows), sink)
        p = sm[0]
        o = p @ v
        dv += p.T @ dout[a:b]
        dp = dout[a:b] @ v.T
        delta = (dout[a:b] * o).sum(axis=1, keepdims=True)
        ds = p * (dp - delta)
        dq[a:b] = scale * (ds @ k)
        dk += scale * (ds.T @ q[a:b])
        if sink is not None:
            dsink -= float((sm[2] * delta[:, 0]).sum())
    if sink is not None:
        return dq, dk, dv, dsink
    return dq, dk, dv


def _check(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("expected [B, H, L, D] arrays")
    B, Hq, _, D = q.shape
    if k.shape[0] != B or v.shape[:3] != k.shape[:3] or k.shape[3] != D:
        raise ValueError("q, k, v shapes disagree")
    Hkv = k.shape[1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return B, Hq, Hkv, Hq // Hkv


def _full_mask(mask, q, k):
    """The mask broadcast (without copying) to [B, Hq, Lq, Lkv], or None."""
    if mask is None:
        return None
    return np.broadcast_to(_mask_values(mask), q.shape[:3] + (k.shape[2],))


def sdpa_forward(q, k, v, scale, is_causal, row_block=None, sinks=None, mask=None):
    """Forward over [B, H, L, D] arrays with GQA ([MLX-VJP] "Key Features").

    Query head h reads KV head h // G with G = Hq // Hkv; ``sinks`` ([Hq] or None) adds
    one sink logit per query head; ``mask`` (broadcastable to [B, Hq, Lq, Lkv], boolean
    or additive, or None) masks scores.  Returns (O [B,Hq,Lq,D], lse [B,Hq,Lq]) in float64.
    """
    B, Hq, Hkv, G = _check(q, k, v)
    mask = _full_mask(mask, q, k)
    o = np.empty(q.shape[:3] + (v.shape[3],))
    lse = np.empty(q.shape[:3])
    for b in range(B):
        for h in range(Hq):
            g = h // G
            o[b, h], lse[b, h] = head_forward(q[b, h], k[b, g], v[b, g], scale,
                                              is_causal, row_block=row_block,
                                              sink=None if sinks is None else float(sinks[h]),
                                              mask=None if mask is None else mask[b, h])
    return o, lse


def group_backward(q, k, v, dout, scale, is_causal, b, g, row_block=None, sinks=None,
                   mask=None):
    """Backward for KV head g of batch b: dQ of its G query heads, and dK, dV of g.

    dK and dV sum the contributions of every query head that reads KV head g
    ([MLX-VJP] "Implementation Notes": several query heads share one KV head).
    Returns (dq [G, Lq, D], dk [Lkv, D], dv [Lkv, D]), and with ``sinks`` also the
    gradients of the group's G sink logits (batch b only).
    """
    B, Hq, Hkv, G = _check(q, k, v)
    mask = _full_mask(mask, q, k)
    dq = np.empty((G,) + q.shape[2:])
    dk = np.zeros(k.shape[2:])
    dv = np.zeros(v.shape[2:])
    dsink = np.zeros(G)
    for t in range(G):
        h = g * G + t
        r = head_backward(q[b, h], k[b, g], v[b, g], dout[b, h], scale, is_causal,
                          row_block=row_block, sink=None if sinks is None else float(sinks[h]),
                          mask=None if mask is None else mask[b, h])
        dq[t], dk_h, dv_h = r[:3]
        if sinks is not None:
            dsink[t] = r[3]
        dk += dk_h
        dv += dv_h
    if sinks is not None:
        return dq, dk, dv, dsink
    return dq, dk, dv


def sdpa_backward(q, k, v, dout, scale, is_causal, row_block=None, sinks=None, mask=None):
    """Backward over [B, H, L, D] arrays.  Returns (dq, dk, dv) in float64, and with
    ``sinks`` ([Hq]) also dsinks [Hq], each summed over the batch.  ``mask``: as in
    sdpa_forward."""
    B, Hq, Hkv, G = _check(q, k, v)
    mask = _full_mask(mask, q, k)
    dq = np.empty(q.shape, dtype=np.float64)
    dk = np.empty(k.shape, dtype=np.float64)
    dv = np.empty(v.shape, dtype=np.float64)
    dsinks = np.zeros(Hq)
    for b in range(B):
        for g in range(Hkv):
            r = group_backward(q, k, v, dout, scale, is_causal, b, g, row_block=row_block,
                               sinks=sinks, mask=mask)
            dq[b, g * G:(g + 1) * G], dk[b, g], dv[b, g] = r[:3]
            if sinks is not None:
                dsinks[g * G:(g + 1) * G] += r[3]
    if sinks is not None:
        return dq, dk, dv, dsinks
    return dq, dk, dv
