"""CPU oracle for fused scaled-dot-product attention: TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check in ``__graft_entry__`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and its
Python binding) never calls it and shares no code with it.
"""
from .ref import (  # noqa: F401
    sdpa_forward,
    sdpa_backward,
    head_forward,
    head_backward,
    group_backward,
)
