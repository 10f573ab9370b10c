"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Covers the five target workloads (the first three in full, the two large ones on whole
sampled (batch, KV-head) groups at full size in the launch configuration the benchmark
times), the test matrix of the MLX VJP work ("[Metal] Add Flash Attention VJP for
training", section "Test Plan": short L for the vector path, longer L for the tiled path,
head dims 32/64/96/128, GQA 4:1, 8:1, 16:1 and MHA, fp16/bf16/fp32, L = 1, non-power-of-2
L, large batch, qL != kvL), every kernel family forced on shapes it serves, determinism
and guard bands around the outputs.
"""
import math

import numpy as np
import pytest
import torch

from parity_util import full_parity, run_gpu, sampled_parity
from scaled_dot_product_flash_gb300 import _lib, api
from scaled_dot_product_flash_gb300.inputs import Shape, draw

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ target workloads
def test_workload_fp32_tiny():
    """fp32, B=1, Hq=Hkv=2, L=64, D=32, non-causal, seed 0."""
    full_parity(Shape(1, 2, 2, 64, 64, 32), "f32", False, seed=0)


def test_workload_fp32_pytensor_shape():
    """fp32, B=8, H=8, L=128, D=64, no mask, seed 1 (the PyTensor issue's timing shape)."""
    full_parity(Shape(8, 8, 8, 128, 128, 64), "f32", False, seed=1)


@pytest.mark.parametrize("causal", [False, True])
def test_workload_fp16_2048(causal):
    """fp16, B=1, H=8, L=2048, D=64, forward and backward, seed 2."""
    full_parity(Shape(1, 8, 8, 2048, 2048, 64), "f16", causal, seed=2)


def test_workload_bf16_gqa_4096_sampled():
    """bf16 GQA 4:1, B=2, Hq=32, Hkv=8, L=4096, D=128, causal, seed 3: full-size run,
    four whole groups checked (two per batch; every query row of their 16 heads,
    the last query block of each batch included, and all keys of their 4 KV heads)."""
    sampled_parity(Shape(2, 32, 8, 4096, 4096, 128), "bf16", True, seed=3,
                   groups=[(0, 0), (0, 5), (1, 2), (1, 7)])


def test_workload_bf16_long_context_sampled():
    """bf16, B=1, H=16, L=16384, D=128, causal, seed 4: full-size run, two heads checked."""
    sampled_parity(Shape(1, 16, 16, 16384, 16384, 128), "bf16", True, seed=4,
                   groups=[(0, 0), (0, 11)])


def test_workload_bf16_head_dim_256_sampled():
    """bf16 GQA 4:1, B=1, Hq=16, Hkv=4, L=4096, D=256, causal, seed 5 (the bench's D = 256
    case): full-size run on the tensor-core kernels, two whole groups checked (the first
    and the last KV head, every query row of their 8 heads)."""
    sampled_parity(Shape(1, 16, 4, 4096, 4096, 256), "bf16", True, seed=5, groups=[(0, 0), (0, 3)])


def test_workload_bf16_short_query():
    """bf16, B=4, Hq=32, Hkv=8, Lq in {1, 4, 8}, Lkv=8192, D=128, non-causal, seed 4:
    drawn one after another from one generator; every output compared."""
    rng = np.random.default_rng(4)
    for lq in (1, 4, 8):
        shape = Shape(4, 32, 8, lq, 8192, 128)
        full_parity(shape, "bf16", False, seed=4, inputs=draw(shape, 4, "bf16", rng=rng))


# ------------------------------------------------------------------ MLX-style matrix
MATRIX = []
for L in (1, 4, 7, 8):          # vector path
    MATRIX.append((Shape(2, 8, 8, L, L, 64), "f16", False))
    MATRIX.append((Shape(2, 8, 2, L, 37, 64), "bf16", True))
for L in (16, 32, 128, 256):    # tiled paths
    MATRIX.append((Shape(2, 8, 8, L, L, 64), "f16", True))
    MATRIX.append((Shape(1, 4, 4, L, L, 128), "bf16", False))
for D in (32, 64, 96, 128):
    for dt in ("f32", "f16", "bf16"):
        MATRIX.append((Shape(1, 4, 2, 100, 100, D), dt, True))
        MATRIX.append((Shape(1, 4, 2, 5, 70, D), dt, False))
for G in (1, 4, 8, 16):
    MATRIX.append((Shape(1, 16, 16 // G, 160, 160, 128), "bf16", True))
    MATRIX.append((Shape(1, 16, 16 // G, 2, 300, 64), "f16", False))
MATRIX += [
    (Shape(1, 2, 1, 1, 1, 64), "bf16", False),           # L = 1
    (Shape(1, 2, 1, 1, 1, 64), "bf16", True),
    (Shape(3, 2, 2, 131, 67, 64), "f16", True),          # qL != kvL, non-power-of-2
    (Shape(1, 2, 2, 67, 131, 128), "bf16", True),
    (Shape(1, 2, 2, 67, 131, 128), "bf16", False),
    (Shape(64, 2, 1, 33, 33, 64), "bf16", True),         # large batch
    (Shape(1, 1, 1, 383, 129, 128), "f32", False),
    (Shape(1, 2, 1, 129, 513, 64), "f16", False),
]


@pytest.mark.parametrize("shape,dtype,causal", MATRIX,
                         ids=[f"{s.B}-{s.Hq}-{s.Hkv}-{s.Lq}-{s.Lkv}-{s.D}-{d}-{'c' if c else 'n'}"
                              for s, d, c in MATRIX])
def test_matrix(shape, dtype, causal):
    full_parity(shape, dtype, causal, seed=100 + shape.Lq + shape.D)


# ------------------------------------------------------------------ bottom-right causal
BOTTOM_RIGHT = [
    (_lib.PATH_AUTO, Shape(1, 8, 2, 200, 700, 128), "bf16"),    # tensor cores, Lq < Lkv
    (_lib.PATH_AUTO, Shape(2, 4, 4, 130, 131, 64), "f16"),      # tensor cores, offset 1
    (_lib.PATH_AUTO, Shape(1, 4, 1, 300, 300, 96), "bf16"),     # tensor cores, Lq = Lkv
    (_lib.PATH_AUTO, Shape(2, 8, 2, 4, 500, 128), "bf16"),      # short query, warp MMA
    (_lib.PATH_AUTO, Shape(1, 4, 2, 40, 130, 32), "f32"),       # CUDA cores
    (_lib.PATH_AUTO, Shape(1, 2, 2, 3, 90, 64), "f32"),         # short query, CUDA cores
    (_lib.PATH_SIMT, Shape(1, 4, 2, 70, 200, 64), "bf16"),      # forced CUDA cores
]


@pytest.mark.parametrize("path,shape,dtype", BOTTOM_RIGHT)
def test_bottom_right_causal(path, shape, dtype):
    """Key j hidden from query i when j > i + Lkv - Lq (the last query sees every key)."""
    with api.force_path(path):
        full_parity(shape, dtype, 2, seed=11)


# ------------------------------------------------------------------ each family forced
FORCED = [
    (_lib.PATH_SIMT, Shape(1, 4, 2, 200, 150, 128), "bf16", True),
    (_lib.PATH_SIMT, Shape(1, 4, 1, 8, 300, 64), "f16", False),
    (_lib.PATH_SIMT, Shape(2, 2, 2, 64, 64, 96), "bf16", False),
    (_lib.PATH_VECTOR, Shape(1, 4, 1, 8, 1000, 128), "bf16", True),
    (_lib.PATH_VECTOR, Shape(2, 8, 2, 8, 513, 32), "f32", False),
    (_lib.PATH_VECTOR, Shape(1, 32, 1, 1, 2000, 96), "f16", False),
    (_lib.PATH_TENSOR, Shape(2, 8, 2, 300, 260, 96), "bf16", True),    # D = 96 on tcgen05
    (_lib.PATH_TENSOR, Shape(1, 4, 4, 257, 129, 96), "f16", False),
    (_lib.PATH_TENSOR, Shape(2, 4, 2, 300, 200, 32), "bf16", True),    # D = 32 on tcgen05
    (_lib.PATH_TENSOR, Shape(1, 2, 2, 140, 390, 32), "f16", False),
]


@pytest.mark.parametrize("path,shape,dtype,causal", FORCED)
def test_forced_family(path, shape, dtype, causal):
    with api.force_path(path):
        full_parity(shape, dtype, causal, seed=7)


def test_vector_threshold_boundary():
    """Lq = 8 takes the vector path, Lq = 9 the tiled path; both agree with the oracle."""
    for lq in (8, 9):
        full_parity(Shape(1, 4, 1, lq, 700, 128), "bf16", False, seed=8)


def test_forced_family_refuses_what_it_cannot_serve():
    q = torch.zeros(1, 4, 64, 64, device="cuda", dtype=torch.bfloat16)
    with api.force_path(_lib.PATH_VECTOR):
        with pytest.raises(_lib.SdpaError) as e:
            api.attention_forward(q, q, q)
        assert e.value.status == 2


# ------------------------------------------------------------------ head dim 256
@pytest.mark.parametrize("shape,dtype,causal", [
    (Shape(1, 2, 1, 40, 70, 256), "f32", True),        # CUDA cores, GQA, ragged
    (Shape(1, 4, 2, 100, 130, 256), "bf16", True),     # 16-bit types also run on CUDA cores
    (Shape(2, 4, 2, 4, 90, 256), "f16", False),        # short query: no short-query kernel
    (Shape(1, 2, 2, 33, 64, 256), "bf16", 2),          # bottom-right causal
])
def test_head_dim_256(shape, dtype, causal):
    full_parity(shape, dtype, causal, seed=31)


@pytest.mark.parametrize("shape,dtype,causal", [
    (Shape(1, 8, 2, 700, 900, 256), "bf16", True),     # several Q tiles, GQA, ragged tails
    (Shape(2, 4, 4, 130, 600, 256), "f16", False),     # five KV tiles: both S buffers reused
    (Shape(1, 4, 1, 257, 257, 256), "bf16", 2),        # bottom-right causal, Lq = Lkv
    (Shape(1, 2, 2, 64, 96, 256), "f16", True),        # one KV tile: the split P path only
])
def test_head_dim_256_on_tensor_cores(shape, dtype, causal):
    """The fp16/bf16 forward and backward at D = 256 on the tensor-core kernels (forced)."""
    with api.force_path(_lib.PATH_TENSOR):
        full_parity(shape, dtype, causal, seed=32)


@pytest.mark.parametrize("shape,dtype,causal", [
    (Shape(1, 4, 1, 200, 330, 256), "bf16", False),    # G = 4: each dK/dV block streams 4 heads
    (Shape(1, 2, 2, 1, 150, 256), "f16", False),       # one query row
    (Shape(1, 2, 1, 100, 300, 256), "bf16", 2),        # bottom-right, offset 200: key tiles start mid-query-range
    (Shape(2, 2, 2, 129, 65, 256), "f16", True),       # top-left causal, one row past a tile
    (Shape(1, 2, 2, 70, 1, 256), "bf16", False),       # a single key
])
def test_head_dim_256_backward_edges(shape, dtype, causal):
    """Edge cases of the D = 256 tensor-core backward: query blocks of 64 rows streamed per
    head of a group, key and query tails, a causal offset, a single key."""
    with api.force_path(_lib.PATH_TENSOR):
        full_parity(shape, dtype, causal, seed=33)


def test_head_dim_256_refusals():
    """The short-query kernels refuse D = 256; the forced tensor path serves the D = 256
    forward and backward, with or without a mask (zero inputs give zero gradients)."""
    q = torch.zeros(1, 2, 4, 256, device="cuda", dtype=torch.bfloat16)
    with api.force_path(_lib.PATH_VECTOR):
        with pytest.raises(_lib.SdpaError) as e:
            api.attention_forward(q, q, q)
        assert e.value.status == 2
    mask = torch.ones(4, 4, dtype=torch.bool, device="cuda")
    with api.force_path(_lib.PATH_TENSOR):
        for m in (None, mask):
            out, lse = api.attention_forward(q, q, q, attn_mask=m)
            dq, dk, dv = api.attention_backward(q, q, q, out, q, lse, attn_mask=m)
            assert torch.count_nonzero(dq) == 0 and torch.count_nonzero(dv) == 0
    api.poll_status()


# ------------------------------------------------------------------ properties
@pytest.mark.parametrize("shape,dtype,causal", [
    (Shape(1, 8, 2, 600, 600, 128), "bf16", True),
    (Shape(2, 8, 2, 4, 900, 64), "f16", False),
    (Shape(1, 2, 2, 100, 100, 64), "f32", True),
    (Shape(1, 8, 2, 300, 460, 256), "bf16", True),  # D = 256: two-CTA partial sums in fixed order
])
def test_bitwise_deterministic(shape, dtype, causal):
    q, k, v, do = draw(shape, 21, dtype)
    a = run_gpu(q, k, v, do, 0.1, causal)
    b = run_gpu(q, k, v, do, 0.1, causal)
    for n in a:
        assert np.array_equal(a[n], b[n]), n


def test_outputs_stay_inside_their_buffers():
    """Guard bands before and after every output keep their canary values."""
    shape = Shape(1, 4, 2, 300, 260, 128)
    q, k, v, do = (t.cuda() for t in draw(shape, 22, "bf16"))
    pad = 4096
    canary = -1536.0  # exactly representable in bf16 and fp32

    def banded(like):
        buf = torch.full((like.numel() + 2 * pad,), canary, device="cuda", dtype=like.dtype)
        return buf, buf[pad:pad + like.numel()].view(like.shape)

    ob, o = banded(q)
    lb, lse = banded(torch.empty(1, 4, 300, device="cuda", dtype=torch.float32))
    api.attention_forward(q, k, v, scale=0.2, is_causal=True, out=o, lse=lse)
    bufs = [banded(q), banded(k), banded(v)]
    api.attention_backward(q, k, v, o, do, lse, scale=0.2, is_causal=True,
                           dq=bufs[0][1], dk=bufs[1][1], dv=bufs[2][1])
    api.poll_status()
    for buf in [ob, lb] + [b for b, _ in bufs]:
        head, tail = buf[:pad].float(), buf[-pad:].float()
        assert bool((head == canary).all()) and bool((tail == canary).all())


def test_lse_is_optional():
    shape = Shape(1, 2, 2, 130, 130, 64)
    q, k, v, _ = (t.cuda() for t in draw(shape, 23, "f16"))
    o1, lse = api.attention_forward(q, k, v, is_causal=True, need_lse=True)
    o2, none = api.attention_forward(q, k, v, is_causal=True, need_lse=False)
    api.poll_status()
    assert none is None
    assert torch.equal(o1, o2)


def test_zero_scale_gives_prefix_means():
    """scale = 0 (uniform attention): O_i is the mean of V over visible keys."""
    shape = Shape(1, 2, 1, 150, 150, 64)
    q, k, v, _ = (t.cuda() for t in draw(shape, 24, "f32"))
    o, lse = api.attention_forward(q, k, v, scale=0.0, is_causal=True)
    api.poll_status()
    ref = v.double().cumsum(2) / torch.arange(1, 151, device="cuda").double()[None, None, :, None]
    assert float((o.double() - ref).abs().max()) < 1e-5
    assert float((lse.double() - torch.log(torch.arange(1, 151, device="cuda").double())).abs().max()) < 1e-5


def test_launch_counter_counts_kernels():
    shape = Shape(1, 2, 2, 64, 64, 64)
    q, k, v, do = (t.cuda() for t in draw(shape, 25, "bf16"))
    n0 = _lib.sdpa_launch_count()
    o, lse = api.attention_forward(q, k, v)
    api.attention_backward(q, k, v, o, do, lse)
    api.poll_status()
    assert _lib.sdpa_launch_count() - n0 >= 3
