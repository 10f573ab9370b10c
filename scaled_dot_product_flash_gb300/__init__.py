"""GB300-native fused scaled-dot-product attention (forward + backward).

The computation lives in ``libsdpa.so`` (hand-written CUDA for sm_103a behind a C ABI,
declared in ``include/sdpa.h``).  This package is its thin Python binding:

* ``_lib``: ctypes entry points under the C names (``sdpa_fwd``, ``sdpa_bwd``, ...).
* ``api``: tensor-level calls that allocate outputs with PyTorch and pass raw pointers.
* ``autograd``: ``SDPAFunction`` (torch autograd over the forward and fused backward) and a
  ``scaled_dot_product_attention`` drop-in for the cases the kernels cover.
* ``inputs``: seeded synthetic inputs.
* ``build``: nvcc build of the library.
"""
from ._lib import (  # noqa: F401
    PATH_AUTO,
    PATH_SIMT,
    PATH_TENSOR,
    PATH_VECTOR,
    SdpaError,
    load,
    sdpa_bwd,
    sdpa_bwd_workspace_size,
    sdpa_fwd,
    sdpa_launch_count,
    sdpa_poll_status,
    sdpa_set_path,
    sdpa_status_string,
)
