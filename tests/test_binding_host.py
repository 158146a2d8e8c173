"""The Python binding refuses inputs its kernels cannot take, before any device
work (no GPU needed): host tensors on the device entry points, unsupported
dtypes and ragged block sizes. There is no CPU fallback to fall into."""

import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import block_sparse_long_bigbird_gb300 as sa  # noqa: E402


def _qkv(dtype=torch.bfloat16, shape=(1, 1, 256, 64)):
    return [torch.zeros(shape, dtype=dtype) for _ in range(3)]


def test_bigbird_fwd_rejects_host_tensors():
    Q, K, V = _qkv()
    table = torch.zeros((1, 4, 3), dtype=torch.int32)
    with pytest.raises(ValueError):
        sa.bigbird_attn_fwd(Q, K, V, 64, 2, 3, 3, table)


def test_longformer_fwd_rejects_host_tensors():
    Q, K, V = _qkv()
    with pytest.raises(ValueError):
        sa.longformer_attn_fwd(Q, K, V, 64, torch.zeros(0, dtype=torch.int32))


def test_backward_rejects_host_tensors():
    Q, K, V = _qkv()
    dO = torch.zeros_like(Q)
    table = torch.zeros((1, 4, 3), dtype=torch.int32)
    with pytest.raises(ValueError):
        sa.bigbird_attn_bwd(Q, K, V, dO, 64, 2, 3, 3, table)
    with pytest.raises(ValueError):
        sa.longformer_attn_bwd(Q, K, V, dO, 64, torch.zeros(0, dtype=torch.int32))


def test_unsupported_dtype_is_a_type_error():
    Q, K, V = _qkv(dtype=torch.float16)
    table = torch.zeros((1, 4, 3), dtype=torch.int32)
    with pytest.raises(TypeError):
        sa.bigbird_attn_fwd(Q, K, V, 64, 2, 3, 3, table)


def test_pattern_builder_needs_whole_blocks():
    with pytest.raises(ValueError):
        sa.build_bigbird_pattern(0, 1, 1000, 64, 2, 3, 3)
    t = sa.build_bigbird_pattern(0, 2, 1024, 64, 2, 3, 3)
    assert t.shape == (2, 16, 3) and t.dtype == torch.int32 and not t.is_cuda
