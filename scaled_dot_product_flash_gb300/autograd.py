"""Autograd integration: a ``torch.autograd.Function`` over the C ABI and a drop-in for
``torch.nn.functional.scaled_dot_product_attention`` restricted to what the kernels do.

The forward keeps the fp32 logsumexp that ``sdpa_fwd`` writes and hands it to
``sdpa_bwd``, which recomputes P from it ("[Metal] Add Flash Attention VJP for training",
sections "Key Features" and "Limitations": the backward needs the forward's logsumexp;
"MPS scaled_dot_product_attention (SDPA)", section "Problem - Unused second output
tensor": the logsumexp is only produced when a gradient will be taken).  As in the rest of
the package, this module only marshals tensors; all arithmetic runs in ``libsdpa.so``.

Supported: q [B, Hq, Lq, D], k and v [B, Hkv, Lkv, D] on CUDA (any layout whose rows are
contiguous, e.g. [B, L, H, D] storage through .transpose(1, 2)), one dtype of fp32/fp16/bf16,
Hq a multiple of Hkv (grouped-query attention: query head h uses KV head h // (Hq/Hkv)),
D in {32, 64, 96, 128, 256}, optional top-left causal mask or ``attn_mask`` (boolean: True keeps
the key; floating: added to the scores; no gradient flows into it), any finite scale,
optional per-head attention-sink logits (``sinks``, differentiable).  Dropout and other
head layouts raise ``NotImplementedError``.
"""
from __future__ import annotations

import math

import torch

from . import api


class SDPAFunction(torch.autograd.Function):
    """out = softmax(scale · q·kᵀ [causal]) · v with a fused backward."""

    @staticmethod
    def forward(ctx, q, k, v, sinks, attn_mask, scale, is_causal):
        needs_grad = any(ctx.needs_input_grad[:4])
        out, lse = api.attention_forward(q, k, v, scale=scale, is_causal=is_causal,
                                         need_lse=needs_grad, sinks=sinks, attn_mask=attn_mask)
        if needs_grad:
            ctx.save_for_backward(q, k, v, out, lse, sinks, attn_mask)
        ctx.scale = scale
        ctx.is_causal = is_causal
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, lse, sinks, attn_mask = ctx.saved_tensors
        if dout.stride(-1) != 1:
            dout = dout.contiguous()
        # The lse already includes the sinks; they are passed only for their own gradient.
        want_ds = sinks is not None and ctx.needs_input_grad[3]
        g = api.attention_backward(q, k, v, out, dout, lse, scale=ctx.scale,
                                   is_causal=ctx.is_causal, sinks=sinks if want_ds else None,
                                   attn_mask=attn_mask)
        return g[0], g[1], g[2], (g[3] if want_ds else None), None, None, None


def scaled_dot_product_attention(query, key, value, attn_mask=None, dropout_p=0.0,
                                 is_causal=False, scale=None, enable_gqa=False, sinks=None):
    """Same call as ``torch.nn.functional.scaled_dot_product_attention`` for the cases the
    kernels cover (see the module docstring); differentiable through ``SDPAFunction``.

    ``is_causal`` is the top-left mask (key j hidden from query i when j > i), as in torch.
    With Hq != Hkv, ``enable_gqa=True`` is required, as in torch.  ``sinks`` (an addition
    to torch's signature): a [Hq] tensor of sink logits, one extra softmax entry per row of
    each query head with a zero value vector; it is used in fp32 and receives a gradient.
    """
    if attn_mask is not None:
        if attn_mask.requires_grad:
            raise NotImplementedError("no gradient is computed for attn_mask")
        if is_causal:
            raise ValueError("attn_mask and is_causal cannot both be set (as in torch)")
    if dropout_p != 0.0:
        raise NotImplementedError("dropout is not supported")
    if query.dim() != 4 or key.dim() != 4 or value.dim() != 4:
        raise NotImplementedError("expected 4-D [B, H, L, D] tensors")
    if key.shape != value.shape:
        raise ValueError("key and value shapes differ")
    B, Hq, Lq, D = query.shape
    Bk, Hkv, Lkv, Dk = key.shape
    if Bk != B or Dk != D:
        raise ValueError("query and key disagree in batch size or head dim")
    if Hq != Hkv and not enable_gqa:
        raise ValueError("Hq != Hkv needs enable_gqa=True")
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    if not (query.dtype == key.dtype == value.dtype):
        raise ValueError("query, key and value must have one dtype")
    if not math.isfinite(1.0 / math.sqrt(D) if scale is None else float(scale)):
        raise ValueError("scale must be finite")
    s = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if sinks is not None:
        if sinks.dim() != 1 or sinks.numel() != Hq:
            raise ValueError("sinks must be a 1-D tensor of Hq sink logits")
        if sinks.device != query.device:
            raise ValueError("sinks must be on the device of query")
        sinks = sinks.to(torch.float32).contiguous()
    # Any layout with contiguous rows is passed through as is (its strides go to the
    # library); others are copied to [B, H, L, D] first.
    q, k, v = (t if t.stride(-1) == 1 else t.contiguous() for t in (query, key, value))
    return SDPAFunction.apply(q, k, v, sinks, attn_mask, s, bool(is_causal))
