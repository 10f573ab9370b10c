"""sdpa_bwd_noalloc: the backward for callers that cannot allocate device memory (a host
application that owns every allocation and passes plugins only their inputs and outputs,
a latency-critical path that must not call cudaMalloc, code running under a locked memory
pool).  Its scratch lives in a static device array inside the library instead of a
caller-provided workspace.  These tests call it through the C ABI and check it against
sdpa_bwd with a workspace, bit for bit, on two calls in a row (the second call finds the first call's
leftovers in the shared array), and check that a problem larger than the array is refused
before anything is launched.  This file sorts last so that a run stopping at the first
failure has already run every other test; it also passes alone in a fresh process."""
import numpy as np
import pytest
import torch

from scaled_dot_product_flash_gb300 import _lib, api
from scaled_dot_product_flash_gb300.inputs import Shape, draw

pytestmark = pytest.mark.gpu


def _run_pair(shape, dtype, causal, seed):
    q, k, v, do = (t.cuda() for t in draw(shape, seed, dtype))
    out, lse = api.attention_forward(q, k, v, is_causal=causal)
    ref = api.attention_backward(q, k, v, out, do, lse, is_causal=causal)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    s = shape
    st = _lib.sdpa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                               do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                               dv.data_ptr(), s.B, s.Hq, s.Hkv, s.Lq, s.Lkv, s.D,
                               1.0 / np.sqrt(s.D), int(causal), api.DTYPE_CODE[q.dtype],
                               torch.cuda.current_stream().cuda_stream)
    assert st == 0, _lib.STATUS_NAMES.get(st, st)
    api.poll_status()
    # The same kernels on the same inputs: the results must be the same bits, so that a
    # stale read from the shared scratch cannot hide inside a tolerance.
    for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert torch.equal(got, want), name
    return dq, dk, dv


def test_noalloc_matches_workspace_backward_twice():
    # First call: a GQA causal problem; second call: a different, smaller problem that
    # reuses the same static scratch (stale contents from the first call in its tail).
    _run_pair(Shape(2, 8, 2, 384, 384, 128), "bf16", True, seed=41)
    _run_pair(Shape(1, 4, 4, 200, 260, 64), "f16", False, seed=42)
    _run_pair(Shape(1, 4, 1, 300, 330, 256), "bf16", True, seed=43)  # D = 256 kernels


def test_noalloc_refuses_problems_larger_than_its_scratch():
    rows = _lib.BWD_NOALLOC_MAX_ROWS
    fake = 0x10000000  # never dereferenced: the size check comes first
    st = _lib.sdpa_bwd_noalloc(fake, fake * 2, fake * 3, fake * 4, fake * 5, fake * 6,
                               fake * 7, fake * 8, fake * 9, 1, 1, 1, rows + 1, 64, 64, 0.125,
                               0, 2, torch.cuda.current_stream().cuda_stream)
    assert st == 5  # SDPA_ERR_WORKSPACE
