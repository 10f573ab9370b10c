"""Tensor-level convenience calls over the C ABI (marshalling only).

PyTorch is used here for device memory and streams: outputs are allocated with torch,
their raw device pointers and the current stream's handle are passed to libsdpa.so, and
a non-OK status is raised as ``SdpaError``.  All arithmetic runs in the library.
"""
from __future__ import annotations

import math

import torch

from . import _lib

DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}

# is_causal values: False/0, True/1 (top-left: key j hidden from query i when j > i) or
# CAUSAL_BOTTOM_RIGHT / "bottom_right" (hidden when j > i + Lkv - Lq; needs Lq <= Lkv).
CAUSAL_NONE, CAUSAL_TOP_LEFT, CAUSAL_BOTTOM_RIGHT = 0, 1, 2


def _causal(c):
    if c is None or c is False:
        return CAUSAL_NONE
    if c is True:
        return CAUSAL_TOP_LEFT
    if c == "bottom_right":
        return CAUSAL_BOTTOM_RIGHT
    if c == "top_left":
        return CAUSAL_TOP_LEFT
    c = int(c)
    if c not in (CAUSAL_NONE, CAUSAL_TOP_LEFT, CAUSAL_BOTTOM_RIGHT):
        raise ValueError(f"is_causal must be False, True or 'bottom_right', not {c}")
    return c


def _check(name, t, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() == 4 and t.stride(-1) != 1:
        raise ValueError(f"{name} must have contiguous rows (stride 1 along D)")
    if t.dim() != 4 and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")


def _layout(t):
    """(batch, head, row) element strides of a [B, H, L, D] tensor: any layout whose rows
    are contiguous, e.g. a [B, L, H, D] buffer seen through .transpose(1, 2)."""
    return (t.stride(0), t.stride(1), t.stride(2))


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dims(q, k):
    B, Hq, Lq, D = q.shape
    Bk, Hkv, Lkv, Dk = k.shape
    if Bk != B or Dk != D:
        raise ValueError("q and k disagree in batch or head dim")
    return B, Hq, Hkv, Lq, Lkv, D


def _check_sinks(name, t, Hq):
    _check(name, t, torch.float32)
    if t.dim() != 1 or t.numel() != Hq:
        raise ValueError(f"{name} must be a 1-D fp32 tensor of Hq = {Hq} sink logits")


def _mask_layout(shape, strides, elem_size, ptr, Lkv):
    """Whether a 4-D mask view (shape, element strides, element size, address) can be
    passed to the library as it is, and its (batch, head, row) strides with 0 for the
    broadcast (size-1) dimensions.  It can if its keys are contiguous and fill whole
    16-byte pieces and every row starts on a 16-byte boundary."""
    direct = (shape[3] == Lkv and strides[3] == 1 and (Lkv * elem_size) % 16 == 0
              and ptr % 16 == 0
              and all(shape[a] == 1 or (strides[a] * elem_size) % 16 == 0 for a in range(3)))
    return direct, tuple(0 if shape[a] == 1 else strides[a] for a in range(3))


def _mask_arg(attn_mask, q, Lq, Lkv):
    """(Mask struct or None, tensor to keep alive) for an attention mask broadcastable to
    [B, Hq, Lq, Lkv]: boolean (True keeps the key) or floating (added to the scores).

    A mask whose rows are 16-byte aligned, with key stride 1 and a key dimension that
    fills whole 16-byte pieces, is passed as a view (broadcast dimensions get stride 0).
    Otherwise its rows are copied into a buffer with the key dimension padded to 16
    bytes (keeping the broadcast dimensions at size 1); the padding is never read as data.
    """
    if attn_mask is None:
        return None, None
    if not attn_mask.is_cuda or attn_mask.device != q.device:
        raise ValueError("attn_mask must be on the device of q")
    if attn_mask.dim() > 4:
        raise ValueError("attn_mask must have at most 4 dimensions")
    m = attn_mask.reshape((1,) * (4 - attn_mask.dim()) + tuple(attn_mask.shape))
    B, Hq = q.shape[0], q.shape[1]
    for size, want, name in zip(m.shape, (B, Hq, Lq, Lkv), ("batch", "head", "query", "key")):
        if size not in (1, want):
            raise ValueError(f"attn_mask {name} dimension {size} does not broadcast to {want}")
    if m.dtype == torch.bool:
        m, kind = m.view(torch.uint8), _lib.MASK_BOOL
    elif m.is_floating_point():
        m, kind = m.to(q.dtype), _lib.MASK_ADDITIVE
    else:
        raise ValueError("attn_mask must be boolean or floating point")
    es = m.element_size()
    direct, strides = _mask_layout(m.shape, m.stride(), es, m.data_ptr(), Lkv)
    if not direct:
        pad = (Lkv * es + 15) // 16 * 16 // es
        buf = torch.zeros(tuple(m.shape[:3]) + (pad,), device=m.device, dtype=m.dtype)
        buf[..., :Lkv] = m
        m = buf
        _, strides = _mask_layout(m.shape, m.stride(), es, m.data_ptr(), pad)
    return _lib.Mask(m.data_ptr(), kind, *strides), m


def attention_forward(q, k, v, scale=None, is_causal=False, need_lse=True, out=None,
                      lse=None, stream=None, sinks=None, attn_mask=None):
    """out = softmax(scale·q·kᵀ [causal]) · v; also the fp32 logsumexp when need_lse.

    q [B,Hq,Lq,D], k/v [B,Hkv,Lkv,D] CUDA tensors of one dtype (fp32/fp16/bf16), in any
    layout with contiguous rows (e.g. [B,L,H,D] storage seen through .transpose(1, 2));
    the strides go to the library, nothing is copied.  `out` defaults to q's layout.
    ``sinks``: optional fp32 [Hq] sink logits, one extra softmax entry per row of each
    query head with a zero value vector (the lse then includes it).  ``attn_mask``:
    optional mask broadcastable to [B, Hq, Lq, Lkv], boolean (True keeps the key) or
    floating (added to the scaled scores); it combines with ``is_causal``.
    Returns (out, lse or None).
    """
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check(n, t, q.dtype)
    B, Hq, Hkv, Lq, Lkv, D = _dims(q, k)
    if v.shape != k.shape:
        raise ValueError("k and v shapes differ")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)  # same layout as q
    if need_lse and lse is None:
        lse = torch.empty((B, Hq, Lq), device=q.device, dtype=torch.float32)
    if not need_lse:
        lse = None
    _check("out", out, q.dtype)
    if sinks is not None:
        _check_sinks("sinks", sinks, Hq)
    strides = _lib.make_strides(q=_layout(q), k=_layout(k), v=_layout(v), o=_layout(out))
    mask, _keep = _mask_arg(attn_mask, q, Lq, Lkv)
    st = _lib.sdpa_fwd_masked(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              lse.data_ptr() if lse is not None else None,
                              sinks.data_ptr() if sinks is not None else None, mask,
                              B, Hq, Hkv, Lq, Lkv, D, scale, _causal(is_causal),
                              DTYPE_CODE[q.dtype], strides, _stream(stream))
    if st != _lib.OK:
        raise _lib.SdpaError(st, "sdpa_fwd")
    return out, lse


def workspace_bytes(q, k):
    B, Hq, Hkv, Lq, Lkv, D = _dims(q, k)
    return _lib.sdpa_bwd_workspace_size(B, Hq, Hkv, Lq, Lkv, D, DTYPE_CODE[q.dtype])


def attention_backward(q, k, v, out, dout, lse, scale=None, is_causal=False, workspace=None,
                       dq=None, dk=None, dv=None, stream=None, sinks=None, dsinks=None,
                       attn_mask=None):
    """(dq, dk, dv) of the forward, from its output ``out`` and logsumexp ``lse``.

    ``attn_mask`` must be the forward's mask (it receives no gradient).

    With ``sinks`` (the forward's fp32 [Hq] sink logits), returns (dq, dk, dv, dsinks),
    dsinks being the fp32 [Hq] gradient of the sink logits summed over the batch.
    """
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out), ("dout", dout)):
        _check(n, t, q.dtype)
    _check("lse", lse, torch.float32)
    B, Hq, Hkv, Lq, Lkv, D = _dims(q, k)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = workspace_bytes(q, k)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check(n, t, q.dtype)
    if sinks is not None:
        _check_sinks("sinks", sinks, Hq)
        dsinks = torch.empty_like(sinks) if dsinks is None else dsinks
        _check_sinks("dsinks", dsinks, Hq)
    elif dsinks is not None:
        raise ValueError("dsinks needs sinks")
    strides = _lib.make_strides(q=_layout(q), k=_layout(k), v=_layout(v), o=_layout(out),
                                dout=_layout(dout), dq=_layout(dq), dk=_layout(dk),
                                dv=_layout(dv))
    mask, _keep = _mask_arg(attn_mask, q, Lq, Lkv)
    st = _lib.sdpa_bwd_masked(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              dout.data_ptr(), lse.data_ptr(),
                              sinks.data_ptr() if sinks is not None else None, mask,
                              dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                              dsinks.data_ptr() if dsinks is not None else None,
                              B, Hq, Hkv, Lq, Lkv, D, scale, _causal(is_causal),
                              DTYPE_CODE[q.dtype], strides, workspace.data_ptr(),
                              workspace.numel(), _stream(stream))
    if st != _lib.OK:
        raise _lib.SdpaError(st, "sdpa_bwd")
    if sinks is not None:
        return dq, dk, dv, dsinks
    return dq, dk, dv


def poll_status(stream=None):
    """Synchronise the stream; raise if a kernel reported a timed-out wait."""
    st = _lib.sdpa_poll_status(_stream(stream))
    if st != _lib.OK:
        raise _lib.SdpaError(st, "sdpa_poll_status")


class force_path:
    """Context manager selecting one kernel family (tests and measurements)."""

    def __init__(self, path: int):
        self.path = path

    def __enter__(self):
        st = _lib.sdpa_set_path(self.path)
        if st != _lib.OK:
            raise _lib.SdpaError(st, "sdpa_set_path")
        return self

    def __exit__(self, *exc):
        _lib.sdpa_set_path(_lib.PATH_AUTO)
        return False
