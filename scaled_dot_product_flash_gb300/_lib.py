"""ctypes binding of libsdpa.so: the C entry points under the same names.

Argument marshalling only.  Every step of the computation runs in the library's CUDA
kernels; there is no fallback of any kind.  If the library has not been built, loading
fails with an error that says how to build it.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsdpa.so")

OK = 0
STATUS_NAMES = {
    0: "SDPA_OK",
    1: "SDPA_ERR_INVALID_ARG",
    2: "SDPA_ERR_UNSUPPORTED",
    3: "SDPA_ERR_CUDA",
    4: "SDPA_ERR_DEVICE_TIMEOUT",
    5: "SDPA_ERR_WORKSPACE",
}
PATH_AUTO, PATH_TENSOR, PATH_SIMT, PATH_VECTOR = 0, 1, 2, 3

# Every symbol include/sdpa.h declares, with its ctypes signature.
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


class Layout(ctypes.Structure):
    """sdpa_layout_t: element strides of the batch, head and row dimensions."""
    _fields_ = [("batch", ctypes.c_int64), ("head", ctypes.c_int64), ("row", ctypes.c_int64)]


class Strides(ctypes.Structure):
    """sdpa_strides_t: one layout per tensor."""
    _fields_ = [(n, Layout) for n in ("q", "k", "v", "o", "dout", "dq", "dk", "dv")]


class Mask(ctypes.Structure):
    """sdpa_mask_t: device pointer, kind and (batch, head, row) element strides."""
    _fields_ = [("ptr", ctypes.c_void_p), ("kind", ctypes.c_int), ("batch", ctypes.c_int64),
                ("head", ctypes.c_int64), ("row", ctypes.c_int64)]


MASK_NONE, MASK_BOOL, MASK_ADDITIVE = 0, 1, 2
_sp = ctypes.POINTER(Strides)
_mp = ctypes.POINTER(Mask)
SIGNATURES = {
    "sdpa_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _vp]),
    "sdpa_bwd_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _i]),
    "sdpa_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                      _i, _i, _i, _i, _i, _i, _f, _i, _i, _vp, _sz, _vp]),
    "sdpa_poll_status": (_i, [_vp]),
    "sdpa_status_string": (ctypes.c_char_p, [_i]),
    "sdpa_set_path": (_i, [_i]),
    "sdpa_launch_count": (ctypes.c_uint64, []),
    "sdpa_timing_enable": (_i, [_i]),
    "sdpa_timing_read": (_i, [_i, ctypes.POINTER(ctypes.c_double),
                              ctypes.POINTER(ctypes.c_uint64)]),
    "sdpa_timing_reset": (None, []),
    "sdpa_debug_inject_timeout": (_i, [_i, ctypes.c_uint64]),
    "sdpa_bwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                              _i, _i, _i, _i, _i, _i, _f, _i, _i, _vp]),
    "sdpa_fwd_strided": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _sp,
                              _vp]),
    "sdpa_bwd_strided": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                              _i, _i, _i, _i, _i, _i, _f, _i, _i, _sp, _vp, _sz, _vp]),
    "sdpa_fwd_sinks": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i,
                            _sp, _vp]),
    "sdpa_bwd_sinks": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                            _i, _i, _i, _i, _i, _i, _f, _i, _i, _sp, _vp, _sz, _vp]),
    "sdpa_fwd_masked": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _mp, _i, _i, _i, _i, _i, _i, _f, _i,
                             _i, _sp, _vp]),
    "sdpa_bwd_masked": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _mp, _vp, _vp, _vp, _vp,
                             _i, _i, _i, _i, _i, _i, _f, _i, _i, _sp, _vp, _sz, _vp]),
}
BWD_NOALLOC_MAX_ROWS = 1 << 20
KERNELS = {"fwd": 0, "delta": 1, "dq": 2, "dkdv": 3, "vec_fwd": 4, "vec_bwd": 5, "sink_grad": 6}

_lib = None


class SdpaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} "
                         f"({status_string(status) if _lib else ''})")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libsdpa.so (once) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it first with "
            "`python -c 'import __graft_entry__ as g; g.build()'` "
            "or `python scaled_dot_product_flash_gb300/build.py`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def sdpa_fwd(q, k, v, out, lse, B, Hq, Hkv, Lq, Lkv, D, scale, is_causal, dtype, stream):
    return load().sdpa_fwd(q, k, v, out, lse, B, Hq, Hkv, Lq, Lkv, D, scale, is_causal,
                           dtype, stream)


def sdpa_bwd_workspace_size(B, Hq, Hkv, Lq, Lkv, D, dtype):
    return load().sdpa_bwd_workspace_size(B, Hq, Hkv, Lq, Lkv, D, dtype)


def sdpa_bwd(q, k, v, out, dout, lse, dq, dk, dv, B, Hq, Hkv, Lq, Lkv, D, scale, is_causal,
             dtype, workspace, workspace_bytes, stream):
    return load().sdpa_bwd(q, k, v, out, dout, lse, dq, dk, dv, B, Hq, Hkv, Lq, Lkv, D, scale,
                           is_causal, dtype, workspace, workspace_bytes, stream)


def make_strides(**layouts) -> Strides:
    """Strides from (batch, head, row) element-stride triples keyed q, k, v, o, dout, dq,
    dk, dv (missing tensors get zeros, which the library rejects if it reads them)."""
    st = Strides()
    for name, (b, h, r) in layouts.items():
        setattr(st, name, Layout(int(b), int(h), int(r)))
    return st


def sdpa_fwd_strided(q, k, v, out, lse, B, Hq, Hkv, Lq, Lkv, D, scale, is_causal, dtype, strides,
                     stream):
    return load().sdpa_fwd_strided(q, k, v, out, lse, B, Hq, Hkv, Lq, Lkv, D, scale, is_causal,
                                   dtype, ctypes.byref(strides), stream)


def sdpa_bwd_strided(q, k, v, out, dout, lse, dq, dk, dv, B, Hq, Hkv, Lq, Lkv, D, scale,
                     is_causal, dtype, strides, workspace, workspace_bytes, stream):
    return load().sdpa_bwd_strided(q, k, v, out, dout, lse, dq, dk, dv, B, Hq, Hkv, Lq, Lkv, D,
                                   scale, is_causal, dtype, ctypes.byref(strides), workspace,
                                   workspace_bytes, stream)


def sdpa_fwd_sinks(q, k, v, out, lse, sinks, B, Hq, Hkv, Lq, Lkv, D, scale, is_causal, dtype,
                   strides, stream):
    """sdpa_fwd_strided with one sink logit per query head (sinks: fp32 [Hq] or None)."""
    return load().sdpa_fwd_sinks(q, k, v, out, lse, sinks, B, Hq, Hkv, Lq, Lkv, D, scale,
                                 is_causal, dtype, ctypes.byref(strides), stream)


def sdpa_bwd_sinks(q, k, v, out, dout, lse, sinks, dq, dk, dv, dsinks, B, Hq, Hkv, Lq, Lkv, D,
                   scale, is_causal, dtype, strides, workspace, workspace_bytes, stream):
    """sdpa_bwd_strided that also writes the sink-logit gradients dsinks (fp32 [Hq])."""
    return load().sdpa_bwd_sinks(q, k, v, out, dout, lse, sinks, dq, dk, dv, dsinks, B, Hq, Hkv,
                                 Lq, Lkv, D, scale, is_causal, dtype, ctypes.byref(strides),
                                 workspace, workspace_bytes, stream)


def sdpa_fwd_masked(q, k, v, out, lse, sinks, mask, B, Hq, Hkv, Lq, Lkv, D, scale, is_causal,
                    dtype, strides, stream):
    """sdpa_fwd_sinks with an attention mask (a ``Mask`` or None)."""
    return load().sdpa_fwd_masked(q, k, v, out, lse, sinks,
                                  ctypes.byref(mask) if mask is not None else None, B, Hq, Hkv,
                                  Lq, Lkv, D, scale, is_causal, dtype, ctypes.byref(strides),
                                  stream)


def sdpa_bwd_masked(q, k, v, out, dout, lse, sinks, mask, dq, dk, dv, dsinks, B, Hq, Hkv, Lq,
                    Lkv, D, scale, is_causal, dtype, strides, workspace, workspace_bytes, stream):
    """sdpa_bwd_sinks with the forward's attention mask (a ``Mask`` or None)."""
    return load().sdpa_bwd_masked(q, k, v, out, dout, lse, sinks,
                                  ctypes.byref(mask) if mask is not None else None, dq, dk, dv,
                                  dsinks, B, Hq, Hkv, Lq, Lkv, D, scale, is_causal, dtype,
                                  ctypes.byref(strides), workspace, workspace_bytes, stream)


def sdpa_bwd_noalloc(q, k, v, out, dout, lse, dq, dk, dv, B, Hq, Hkv, Lq, Lkv, D, scale,
                     is_causal, dtype, stream):
    """sdpa_bwd with its scratch in the library's static device array (no workspace)."""
    return load().sdpa_bwd_noalloc(q, k, v, out, dout, lse, dq, dk, dv, B, Hq, Hkv, Lq, Lkv, D,
                                   scale, is_causal, dtype, stream)


def sdpa_poll_status(stream):
    return load().sdpa_poll_status(stream)


def status_string(status: int) -> str:
    return load().sdpa_status_string(status).decode()


def sdpa_status_string(status: int) -> str:
    return status_string(status)


def sdpa_set_path(path: int) -> int:
    return load().sdpa_set_path(path)


def sdpa_launch_count() -> int:
    return int(load().sdpa_launch_count())


def sdpa_timing_enable(on: bool) -> int:
    return load().sdpa_timing_enable(int(bool(on)))


def sdpa_timing_read(kernel: int):
    """(total_ms, launches) of one kernel kind since the last reset."""
    ms = ctypes.c_double(0.0)
    n = ctypes.c_uint64(0)
    st = load().sdpa_timing_read(kernel, ctypes.byref(ms), ctypes.byref(n))
    if st != OK:
        raise SdpaError(st, "sdpa_timing_read")
    return ms.value, int(n.value)


def sdpa_timing_reset() -> None:
    load().sdpa_timing_reset()


def sdpa_debug_inject_timeout(on: bool, wait_limit_ns: int) -> int:
    return load().sdpa_debug_inject_timeout(int(bool(on)), int(wait_limit_ns))
