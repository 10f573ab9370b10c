"""Failure detection without a GPU fault: a kernel wait that can never complete must run
out of its time limit, record SDPA_ERR_DEVICE_TIMEOUT in the device error word and return,
leaving the CUDA context usable.  The failure is planted from the host: the test hook makes
the next tensor-core forward withhold its first K tile (a flag that nothing ever sets)."""
import pytest
import torch

from scaled_dot_product_flash_gb300 import _lib, api
from scaled_dot_product_flash_gb300.inputs import Shape, draw

pytestmark = pytest.mark.gpu

DEFAULT_LIMIT_NS = 2_000_000_000


def test_withheld_tile_times_out_and_is_reported():
    q, k, v, _ = (t.cuda() for t in draw(Shape(1, 2, 2, 256, 256, 128), 31, "bf16"))
    assert _lib.sdpa_debug_inject_timeout(True, 200_000_000) == 0
    try:
        with api.force_path(_lib.PATH_TENSOR):
            api.attention_forward(q, k, v)
        st = _lib.sdpa_poll_status(torch.cuda.current_stream().cuda_stream)
        assert st == 4, _lib.STATUS_NAMES.get(st, st)   # SDPA_ERR_DEVICE_TIMEOUT
        # The error word was cleared by the poll, and the context still works.
        assert _lib.sdpa_poll_status(torch.cuda.current_stream().cuda_stream) == 0
    finally:
        _lib.sdpa_debug_inject_timeout(False, DEFAULT_LIMIT_NS)
    out, lse = api.attention_forward(q, k, v)
    api.poll_status()
    ref, _ = api.attention_forward(q.float(), k.float(), v.float())
    api.poll_status()
    assert float((out.float() - ref).abs().max()) < 8e-3


def test_hook_rejects_zero_limit():
    assert _lib.sdpa_debug_inject_timeout(False, 0) == 1
