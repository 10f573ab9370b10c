"""C-ABI checks that need no GPU: the library loads, exports every declared symbol, and
rejects bad arguments on the host with the documented status codes before any launch."""
import ctypes
import os
import re

import pytest

from scaled_dot_product_flash_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdpa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sdpa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_documented_calls():
    names = declared_functions()
    for n in ("sdpa_fwd", "sdpa_bwd", "sdpa_bwd_workspace_size", "sdpa_poll_status",
              "sdpa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    for code in range(6):
        assert _lib.status_string(code) not in ("", "unknown status")
    assert _lib.status_string(99) == "unknown status"


def test_workspace_size(lib):
    # fp32 delta per query row, rounded up to 256 bytes
    assert _lib.sdpa_bwd_workspace_size(2, 32, 8, 4096, 4096, 128, 2) == 2 * 32 * 4096 * 4
    assert _lib.sdpa_bwd_workspace_size(1, 1, 1, 1, 1, 64, 0) == 256
    assert _lib.sdpa_bwd_workspace_size(1, 3, 2, 8, 8, 64, 0) == 0   # Hq % Hkv != 0
    assert _lib.sdpa_bwd_workspace_size(1, 2, 2, 8, 8, 48, 0) == 0   # unsupported D


# Fake, 16-byte aligned, non-overlapping "device" addresses: every case below must be
# rejected by host-side validation, so nothing is ever dereferenced or launched.
Q, K, V, O, L, DO, DQ, DK, DV, WS = (0x10000000 * (n + 1) for n in range(10))
GOOD = dict(B=1, Hq=2, Hkv=1, Lq=64, Lkv=64, D=64, scale=0.125, causal=0, dtype=2)


def fwd(lib, q=Q, k=K, v=V, o=O, lse=L, **kw):
    a = dict(GOOD, **kw)
    return _lib.sdpa_fwd(q, k, v, o, lse, a["B"], a["Hq"], a["Hkv"], a["Lq"], a["Lkv"], a["D"],
                         a["scale"], a["causal"], a["dtype"], None)


def bwd(lib, ws=WS, ws_bytes=1 << 20, dq=DQ, lse=L, **kw):
    a = dict(GOOD, **kw)
    return _lib.sdpa_bwd(Q, K, V, O, DO, lse, dq, DK, DV, a["B"], a["Hq"], a["Hkv"], a["Lq"],
                         a["Lkv"], a["D"], a["scale"], a["causal"], a["dtype"], ws, ws_bytes,
                         None)


INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 5


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), INVALID),
    (dict(o=0), INVALID),
    (dict(k=K + 8), INVALID),                 # misaligned
    (dict(lse=L + 4), INVALID),               # misaligned
    (dict(B=0), INVALID),
    (dict(Lq=0), INVALID),
    (dict(Lkv=0), INVALID),
    (dict(Hq=3, Hkv=2), INVALID),             # Hq % Hkv
    (dict(scale=float("nan")), INVALID),
    (dict(scale=float("inf")), INVALID),
    (dict(D=48), UNSUPPORTED),
    (dict(D=512), UNSUPPORTED),
    (dict(dtype=3), UNSUPPORTED),
    (dict(B=70000), UNSUPPORTED),
    (dict(o=Q + 64), INVALID),                # out overlaps q
    (dict(lse=O), INVALID),                   # lse overlaps out
    (dict(causal=3), INVALID),                # unknown causal mode
    (dict(causal=-1), INVALID),
    (dict(causal=2, Lq=65, Lkv=64), UNSUPPORTED),   # bottom-right needs Lq <= Lkv
])
def test_forward_rejects(lib, kw, code):
    assert fwd(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(ws=0), WORKSPACE),
    (dict(ws_bytes=100), WORKSPACE),
    (dict(lse=0), INVALID),
    (dict(dq=Q), INVALID),                    # dq aliases q
    (dict(dq=DQ + 2), INVALID),
    (dict(ws=DK), INVALID),                   # workspace overlaps dk
    (dict(Hq=4, Hkv=3), INVALID),
    (dict(D=80), UNSUPPORTED),
])
def test_backward_rejects(lib, kw, code):
    assert bwd(lib, **kw) == code


def test_set_path(lib):
    assert _lib.sdpa_set_path(7) == INVALID
    assert _lib.sdpa_set_path(-1) == INVALID
    for p in (_lib.PATH_TENSOR, _lib.PATH_SIMT, _lib.PATH_VECTOR, _lib.PATH_AUTO):
        assert _lib.sdpa_set_path(p) == 0


def test_launch_counter_is_readable(lib):
    assert isinstance(_lib.sdpa_launch_count(), int)


def test_product_path_has_no_oracle_dependency():
    """The library binding and the CUDA sources never touch the oracle package."""
    pkg = os.path.join(ROOT, "scaled_dot_product_flash_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\b(import|from)\s+oracle\b|oracle[./]", text), f


# ---- strided entry points: every case below is rejected before anything is launched.
def _cont(H, L, D):
    return (H * L * D, L * D, D)


def fwd_strided(lib, out_ptr=O, **lay):
    a = GOOD
    B, Hq, Hkv, Lq, Lkv, D = a["B"], a["Hq"], a["Hkv"], a["Lq"], a["Lkv"], a["D"]
    layouts = dict(q=_cont(Hq, Lq, D), k=_cont(Hkv, Lkv, D), v=_cont(Hkv, Lkv, D),
                   o=_cont(Hq, Lq, D))
    layouts.update(lay)
    st = _lib.make_strides(**layouts)
    return _lib.sdpa_fwd_strided(Q, K, V, out_ptr, L, B, Hq, Hkv, Lq, Lkv, D, a["scale"],
                                 a["causal"], a["dtype"], st, None)


@pytest.mark.parametrize("kw", [
    dict(q=(8192, 4096, 65)),          # row stride not a multiple of 16 bytes
    dict(q=(8192, 4096, 32)),          # rows overlap (row stride < D)
    dict(k=(4096, 0, 64)),             # zero stride
    dict(v=(4096, 4096, -64)),         # negative stride
    dict(q=(8192, 64, 64)),            # heads and rows share addresses
    dict(o=(8192, 64, 128), q=(8192, 64, 128)),     # [B, L, H, D] out at q's address: overlap
])
def test_forward_strided_rejects(lib, kw):
    out_ptr = Q + 16 if "o" in kw else O
    assert fwd_strided(lib, out_ptr=out_ptr, **kw) == INVALID


def test_strided_null_strides_rejected(lib):
    a = GOOD
    assert lib.sdpa_fwd_strided(Q, K, V, O, L, a["B"], a["Hq"], a["Hkv"], a["Lq"], a["Lkv"],
                                a["D"], a["scale"], a["causal"], a["dtype"], None, None) == INVALID


# ---- sink entry points: every case below is rejected before anything is launched.
SK, DSK = 0x10000000 * 11, 0x10000000 * 12


def _all_cont():
    a = GOOD
    q = _cont(a["Hq"], a["Lq"], a["D"])
    k = _cont(a["Hkv"], a["Lkv"], a["D"])
    return _lib.make_strides(q=q, k=k, v=k, o=q, dout=q, dq=q, dk=k, dv=k)


def fwd_sinks(sinks):
    a = GOOD
    return _lib.sdpa_fwd_sinks(Q, K, V, O, L, sinks, a["B"], a["Hq"], a["Hkv"], a["Lq"],
                               a["Lkv"], a["D"], a["scale"], a["causal"], a["dtype"], _all_cont(),
                               None)


def bwd_sinks(sinks, dsinks):
    a = GOOD
    return _lib.sdpa_bwd_sinks(Q, K, V, O, DO, L, sinks, DQ, DK, DV, dsinks, a["B"], a["Hq"],
                               a["Hkv"], a["Lq"], a["Lkv"], a["D"], a["scale"], a["causal"],
                               a["dtype"], _all_cont(), WS, 1 << 20, None)


@pytest.mark.parametrize("sinks", [SK + 2, O + 64, L + 4])   # misaligned, in out, in lse
def test_forward_sinks_rejects(lib, sinks):
    assert fwd_sinks(sinks) == INVALID


@pytest.mark.parametrize("sinks,dsinks", [
    (None, DSK),          # a sink gradient without sinks
    (SK, DSK + 1),        # misaligned
    (SK, DQ + 16),        # dsinks inside dq
    (SK, SK),             # dsinks aliases sinks
    (SK, L + 8),          # dsinks inside lse
    (SK + 2, DSK),        # misaligned sinks
    (WS + 4, DSK),        # sinks inside the workspace
])
def test_backward_sinks_rejects(lib, sinks, dsinks):
    assert bwd_sinks(sinks, dsinks) == INVALID


# ---- masked entry points: every case below is rejected before anything is launched.
MK = 0x10000000 * 13


def fwd_masked(ptr=MK, kind=1, batch=0, head=0, row=64):
    a = GOOD
    m = _lib.Mask(ptr, kind, batch, head, row)
    return _lib.sdpa_fwd_masked(Q, K, V, O, L, None, m, a["B"], a["Hq"], a["Hkv"], a["Lq"],
                                a["Lkv"], a["D"], a["scale"], a["causal"], a["dtype"],
                                _all_cont(), None)


@pytest.mark.parametrize("kw", [
    dict(kind=3),                  # unknown kind
    dict(kind=-1),
    dict(ptr=0),                   # no pointer with a mask kind
    dict(ptr=MK + 8),              # misaligned
    dict(row=8),                   # bool row stride of 8 bytes
    dict(kind=2, row=4),           # additive bf16 row stride of 8 bytes
    dict(head=-64),                # negative stride
    dict(ptr=O + 4096),            # inside out
    dict(ptr=L),                   # inside lse
])
def test_forward_masked_rejects(lib, kw):
    assert fwd_masked(**kw) == INVALID


def test_backward_masked_rejects_a_mask_inside_an_output(lib):
    a = GOOD
    m = _lib.Mask(DK + 1024, 1, 0, 0, 64)
    assert _lib.sdpa_bwd_masked(Q, K, V, O, DO, L, None, m, DQ, DK, DV, None, a["B"], a["Hq"],
                                a["Hkv"], a["Lq"], a["Lkv"], a["D"], a["scale"], a["causal"],
                                a["dtype"], _all_cont(), WS, 1 << 20, None) == INVALID
