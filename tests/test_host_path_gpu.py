"""The host-buffer entry points (copies pipelined against the computation)
give bitwise the results of the device entry points."""

import numpy as np
import pytest
import torch

import block_sparse_long_bigbird_gb300 as sa
from block_sparse_long_bigbird_gb300.inputs import make_key_mask, make_qkv
from parity_util import pattern_table

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,n,d,b,padded", [(2, 3, 1024, 64, 64, False), (1, 16, 2048, 128, 128, True),
                                              (3, 12, 512, 64, 64, True)])
def test_bigbird_host_path_matches_device_path(B, H, n, d, b, padded):
    dev = torch.device("cuda:0")
    g, w, r = 2, 3, 3
    Q, K, V = make_qkv(B, H, n, d, "bf16", cfg_id=96)
    table = pattern_table(0, H, n, b, g, w, r)
    km = make_key_mask(B, n) if padded else None
    ref = sa.bigbird_attn_fwd(Q.to(dev), K.to(dev), V.to(dev), b, g, w, r, table.to(dev),
                              None if km is None else km.to(dev)).cpu()
    Qh, Kh, Vh = (t.pin_memory() for t in (Q, K, V))
    for _ in range(3):  # repeated calls reuse the staging sets
        out = sa.bigbird_attn_fwd_host(Qh, Kh, Vh, b, g, w, r, table, km)
        torch.cuda.synchronize()
        assert sa.get_last_device_status() == 0
        assert torch.equal(out, ref)


def test_longformer_host_path_matches_device_path_pageable():
    dev = torch.device("cuda:0")
    B, H, n, d = 2, 4, 1000, 64
    Q, K, V = make_qkv(B, H, n, d, "bf16", cfg_id=97)
    gidx = torch.tensor([0, 5, 500], dtype=torch.int32)
    dil = torch.tensor([0, 1, 0, 2], dtype=torch.int32)
    km = make_key_mask(B, n)
    ref = sa.longformer_attn_fwd(Q.to(dev), K.to(dev), V.to(dev), 128, gidx.to(dev), km.to(dev),
                                 dilation=dil.to(dev), causal=True).cpu()
    out = torch.empty_like(Q)  # pageable output: copies do not overlap but results are the same
    sa.longformer_attn_fwd_host(Q, K, V, 128, gidx, km, out=out, dilation=dil, causal=True)
    torch.cuda.synchronize()
    assert sa.get_last_device_status() == 0
    assert torch.equal(out, ref)


def test_host_path_fp32():
    dev = torch.device("cuda:0")
    B, H, n, d, b, g, w, r = 1, 2, 1024, 64, 64, 2, 3, 3
    Q, K, V = make_qkv(B, H, n, d, "fp32", cfg_id=98)
    table = pattern_table(0, H, n, b, g, w, r)
    ref = sa.bigbird_attn_fwd(Q.to(dev), K.to(dev), V.to(dev), b, g, w, r, table.to(dev)).cpu()
    out = sa.bigbird_attn_fwd_host(Q.pin_memory(), K.pin_memory(), V.pin_memory(), b, g, w, r, table)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


@pytest.mark.parametrize("B", [1, 3])
def test_longformer_host_path_residue_classes(B):
    # Dilated heads, no global tokens, no padding: every chunk of the host path
    # (heads of one entry for B = 1, whole entries for B = 3) runs its dilated
    # heads on residue-class copies, with its slice of the dilation array.
    dev = torch.device("cuda:0")
    H, n, d = 8, 2400, 64
    Q, K, V = make_qkv(B, H, n, d, "bf16", cfg_id=99)
    dil = torch.tensor([0, 3, 1, 2, 0, 3, 6, 1], dtype=torch.int32)  # stride 7 does not divide 2400: direct path
    ref = sa.longformer_attn_fwd(Q.to(dev), K.to(dev), V.to(dev), 256, None, None,
                                 dilation=dil.to(dev), causal=True).cpu()
    Qh, Kh, Vh = (t.pin_memory() for t in (Q, K, V))
    out = sa.longformer_attn_fwd_host(Qh, Kh, Vh, 256, None, None, dilation=dil, causal=True)
    torch.cuda.synchronize()
    assert sa.get_last_device_status() == 0
    assert torch.equal(out, ref)
