"""Host-side argument handling of the Python API that needs no GPU: how masks are laid out
for the library, and the checks that run before anything reaches it."""
import pytest
import torch

from scaled_dot_product_flash_gb300 import api


@pytest.mark.parametrize("shape,strides,es,ptr,lkv,direct,want", [
    ((1, 1, 128, 64), (8192, 8192, 64, 1), 1, 4096, 64, True, (0, 0, 64)),          # shared bool
    ((2, 1, 1, 100), (100, 100, 100, 1), 1, 4096, 100, False, (100, 0, 0)),         # 100 B rows
    ((1, 4, 32, 64), (8192, 2048, 64, 1), 2, 4096, 64, True, (0, 2048, 64)),        # per-head f16
    ((2, 4, 32, 64), (8192, 2048, 64, 1), 2, 4104, 64, False, (8192, 2048, 64)),    # misaligned
    ((1, 1, 32, 64), (2048, 2048, 1, 32), 2, 4096, 64, False, (0, 0, 1)),           # keys strided
    ((1, 1, 32, 1), (32, 32, 1, 1), 2, 4096, 64, False, (0, 0, 1)),                 # keys broadcast
    ((3, 1, 1, 64), (64, 64, 64, 1), 1, 4096, 64, True, (64, 0, 0)),                # key padding
    ((3, 1, 1, 64), (72, 64, 64, 1), 1, 4096, 64, False, (72, 0, 0)),               # 72 B batch step
])
def test_mask_layout(shape, strides, es, ptr, lkv, direct, want):
    assert api._mask_layout(shape, strides, es, ptr, lkv) == (direct, want)


def test_padded_copy_layout_is_direct():
    """The padded buffer the API builds for a non-direct mask always qualifies."""
    for lkv, es in ((77, 1), (100, 2), (260, 2), (31, 4)):
        pad = (lkv * es + 15) // 16 * 16 // es
        buf = torch.zeros(2, 1, 5, pad)
        strides = buf.stride()
        direct, _ = api._mask_layout((2, 1, 5, pad), strides, es, 4096, pad)
        assert direct and (pad * es) % 16 == 0 and pad >= lkv


def test_mask_on_the_host_is_rejected():
    q = torch.zeros(1, 2, 8, 32)
    with pytest.raises(ValueError):
        api._mask_arg(torch.ones(8, 8, dtype=torch.bool), q, 8, 8)


def test_causal_modes():
    assert api._causal(False) == api.CAUSAL_NONE
    assert api._causal(True) == api.CAUSAL_TOP_LEFT
    assert api._causal("bottom_right") == api.CAUSAL_BOTTOM_RIGHT
    with pytest.raises(ValueError):
        api._causal(3)
