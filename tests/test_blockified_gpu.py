"""The pages' dense-operation formulation (``baselines.blockified``) on the GPU,
at the library's workload shapes and dtypes, against the float64 oracle.

This is the comparison baseline that ``bench.py --impl blockified`` times; the
check here makes sure that what is timed computes the same function, within
the same tolerances the library is held to.
"""

import numpy as np
import pytest
import torch

from baselines.blockified import bigbird_blockified, longformer_chunks
from block_sparse_long_bigbird_gb300.inputs import make_key_mask, make_qkv
from block_sparse_long_bigbird_gb300.workloads import WORKLOADS
from oracle import bigbird_random_table, oracle_bigbird, oracle_longformer
from parity_util import assert_close, sampled_bigbird_rows

pytestmark = pytest.mark.gpu


def _bigbird(wl, heads, rows=None):
    dev = torch.device("cuda:0")
    Q, K, V = make_qkv(wl.B, wl.H, wl.n, wl.d, wl.dtype, sigma=wl.sigma, cfg_id=wl.cfg_id)
    table = bigbird_random_table(wl.seed, wl.H, wl.n, wl.b, wl.g, wl.w, wl.r)
    km = make_key_mask(wl.B, wl.n) if wl.padded else None
    O = bigbird_blockified(Q.to(dev), K.to(dev), V.to(dev), wl.b, wl.g, wl.w, wl.r,
                           torch.from_numpy(table).to(dev), None if km is None else km.to(dev))
    O = O.float().cpu().numpy()
    for beta, h in heads:
        sl = (slice(beta, beta + 1), slice(h, h + 1))
        ref = oracle_bigbird(Q[sl], K[sl], V[sl], wl.b, wl.g, wl.w, table[h:h + 1],
                             key_mask=None if km is None else km[beta:beta + 1].numpy(), rows=rows)[0, 0]
        got = O[beta, h] if rows is None else O[beta, h][rows]
        assert_close(got, ref, wl.tol_max, wl.tol_mean, what=f"{wl.name} beta={beta} h={h}")


def test_bigbird_blockified_fp32_n1024():
    _bigbird(WORKLOADS["bigbird_fp32_n1024"], [(0, 0)])


def test_bigbird_blockified_bf16_n4096():
    _bigbird(WORKLOADS["bigbird_bf16_n4096"], [(0, 0), (3, 7), (7, 11)])


def test_bigbird_blockified_padded_n16384():
    wl = WORKLOADS["bigbird_bf16_n16384_padded"]
    _bigbird(wl, [(0, 3), (1, 15)], rows=sampled_bigbird_rows(wl.n, wl.b, wl.g, n_random_blocks=6, seed=4))


def test_bigbird_blockified_d128_n65536():
    wl = WORKLOADS["bigbird_bf16_n65536_d128"]
    _bigbird(wl, [(0, 5)], rows=sampled_bigbird_rows(wl.n, wl.b, wl.g, n_random_blocks=4, seed=5))


def test_longformer_chunks_bf16_n4096():
    wl = WORKLOADS["longformer_bf16_n4096"]
    dev = torch.device("cuda:0")
    Q, K, V = make_qkv(wl.B, wl.H, wl.n, wl.d, wl.dtype, cfg_id=wl.cfg_id)
    gidx = np.arange(wl.n_global)
    O = longformer_chunks(Q.to(dev), K.to(dev), V.to(dev), wl.window, torch.from_numpy(gidx).to(dev))
    O = O.float().cpu().numpy()
    for beta, h in [(0, 0), (3, 11)]:
        sl = (slice(beta, beta + 1), slice(h, h + 1))
        ref = oracle_longformer(Q[sl], K[sl], V[sl], wl.window, gidx)[0, 0]
        assert_close(O[beta, h], ref, wl.tol_max, wl.tol_mean, what=f"longformer beta={beta} h={h}")
