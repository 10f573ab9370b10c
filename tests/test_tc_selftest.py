"""GPU unit test of the tcgen05 building blocks the tensor-core kernels are made of:
TMA loads with 128-byte swizzle, shared-memory descriptors for K-major and MN-major
operands, the f16-kind instruction descriptor, A operands in tensor memory, and TMEM
loads.  Each variant is a 128x128x128 bf16 product checked against a CPU matmul."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def selftest_lib():
    out = os.path.join(ROOT, "_build", "libtcselftest.so")
    src = os.path.join(ROOT, "tests", "tc_selftest.cu")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                    "-Xcompiler", "-fPIC", "-shared", "-o", out, src], check=True)
    lib = ctypes.CDLL(out)
    lib.selftest_mma.restype = ctypes.c_int
    lib.selftest_mma.argtypes = [ctypes.c_int] + [ctypes.c_void_p] * 4
    return lib


@pytest.mark.parametrize("variant", [0, 1, 2])
def test_mma_variant(selftest_lib, variant):
    g = torch.Generator().manual_seed(variant)
    a = torch.randn(128, 128, generator=g).to(torch.bfloat16)
    b = torch.randn(128, 128, generator=g).to(torch.bfloat16)
    ad, bd = a.cuda(), b.cuda()
    out = torch.zeros(128, 128, device="cuda", dtype=torch.float32)
    err = torch.zeros(1, device="cuda", dtype=torch.int32)
    rc = selftest_lib.selftest_mma(variant, ad.data_ptr(), bd.data_ptr(), out.data_ptr(),
                                   err.data_ptr())
    assert rc == 0
    assert int(err.item()) == 0
    a64, b64 = a.double().numpy(), b.double().numpy()
    ref = a64 @ b64.T if variant == 0 else a64 @ b64
    np.testing.assert_allclose(out.double().cpu().numpy(), ref, atol=1e-3, rtol=1e-4)
