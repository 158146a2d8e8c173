"""The pages' dense-operation formulation (``baselines.blockified``) against the
float64 oracle on the CPU.

Run in float64, the blockified products must give the oracle's masked dense
softmax up to rounding: "Big Bird", App. D (Fig. 6 caption) has the dense
product over the blocked queries and the concatenated K'' equal the sparse
pattern of its Fig. 3(d), and "Longformer", App. A has the chunks version
compute the same banded product as its loop version. The cases cover global,
window and random blocks at the sequence ends (where a rolled copy wraps and
must be masked), a window block that is also global, key padding, a pattern
with no random or global blocks, Longformer chunks with and without global
tokens, a window wider than the sequence, padding and autoregressive mode.
"""

import numpy as np
import pytest
import torch

from baselines.blockified import bigbird_blockified, longformer_chunks
from block_sparse_long_bigbird_gb300.inputs import make_key_mask, make_qkv
from oracle import bigbird_random_table, oracle_bigbird, oracle_longformer

EXACT = 1e-12


@pytest.mark.parametrize("B,H,n,d,b,g,w,r,pad", [
    (1, 1, 1024, 64, 64, 2, 3, 3, False),   # the small fp32 workload's pattern
    (2, 2, 512, 32, 32, 1, 5, 2, True),     # key padding, wider window
    (1, 2, 768, 16, 64, 3, 7, 4, False),    # window blocks that are global (j - 3 < g)
    (1, 1, 256, 8, 32, 0, 3, 0, True),      # window only, padded
    (1, 1, 256, 8, 32, 2, 1, 2, False),     # window of one block
    (1, 1, 128, 8, 32, 2, 3, 3, False),     # g + w covers every block: full attention
])
def test_bigbird_blockified_equals_the_oracle(B, H, n, d, b, g, w, r, pad):
    Q, K, V = (x.double() for x in make_qkv(B, H, n, d, "fp32", cfg_id=90))
    table = bigbird_random_table(0, H, n, b, g, w, r)
    km = make_key_mask(B, n, seed=7) if pad else None
    got = bigbird_blockified(Q, K, V, b, g, w, r, torch.from_numpy(table), km).numpy()
    ref = oracle_bigbird(Q, K, V, b, g, w, table, key_mask=None if km is None else km.numpy())
    assert np.abs(got - ref).max() <= EXACT


def test_bigbird_blockified_attends_a_repeated_random_block_once():
    # A caller's table may repeat a block, or name a window or global block: the
    # oracle's mask is a set, so each key is attended once.
    B, H, n, d, b, g, w = 1, 1, 512, 16, 32, 2, 3
    Q, K, V = (x.double() for x in make_qkv(B, H, n, d, "fp32", cfg_id=91))
    nb = n // b
    table = np.full((H, nb, 3), -1, dtype=np.int32)
    for j in range(g, nb):
        table[0, j] = [(j + 5) % nb, (j + 5) % nb, min(j + 1, nb - 1)]  # repeat; a window block
    got = bigbird_blockified(Q, K, V, b, g, w, 3, torch.from_numpy(table)).numpy()
    ref = oracle_bigbird(Q, K, V, b, g, w, table)
    assert np.abs(got - ref).max() <= EXACT


@pytest.mark.parametrize("B,H,n,d,window,ng,pad,causal", [
    (1, 2, 1000, 16, 64, 5, False, False),   # n not a multiple of window / 2
    (2, 1, 512, 8, 32, 0, True, False),      # no global tokens, padded
    (1, 1, 300, 8, 16, 3, True, True),       # autoregressive, padded
    (1, 1, 4096, 8, 512, 16, False, False),  # the n = 4096 Longformer pattern
    (1, 1, 96, 8, 256, 2, False, False),     # window wider than the sequence
])
def test_longformer_chunks_equal_the_oracle(B, H, n, d, window, ng, pad, causal):
    Q, K, V = (x.double() for x in make_qkv(B, H, n, d, "fp32", cfg_id=92))
    gidx = np.sort(np.random.default_rng(1).choice(n, ng, replace=False)) if ng else np.zeros(0, np.int64)
    km = make_key_mask(B, n, seed=8) if pad else None
    got = longformer_chunks(Q, K, V, window, torch.from_numpy(gidx), km, causal=causal).numpy()
    ref = oracle_longformer(Q, K, V, window, gidx, key_mask=None if km is None else km.numpy(), causal=causal)
    assert np.abs(got - ref).max() <= EXACT


def test_blockified_imports_nothing_from_the_library():
    import ast
    import pathlib

    src = pathlib.Path(__file__).resolve().parent.parent / "baselines" / "blockified.py"
    mods = set()
    for node in ast.walk(ast.parse(src.read_text())):
        if isinstance(node, ast.Import):
            mods |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom):
            mods.add((node.module or "").split(".")[0])
    assert mods <= {"math", "torch"}, mods
