"""Seeded random sweeps of small shapes through the tensor-core path, every row
compared with the float64 oracle (the oracle drawing its own pattern table).

Each case draws its sizes and pattern parameters from a fixed seed, so a
failure names a reproducible case: BigBird over b, d, g, w, r and prefix or
random key padding; Longformer over ragged n, window widths (0 up to wider
than n), global positions, per-head dilation, the autoregressive mode and
padding (with and without global tokens, so both the direct dilated path and
the residue-class copies run).
"""

import numpy as np
import pytest
import torch

from block_sparse_long_bigbird_gb300.inputs import make_global_positions, make_key_mask, make_random_key_mask
from parity_util import bigbird_case, longformer_case

pytestmark = pytest.mark.gpu


def _bigbird_params(seed):
    rng = np.random.default_rng(1000 + seed)
    b = int(rng.choice([64, 128]))
    d = int(rng.choice([64, 128]))
    nb = int(rng.integers(2, 17))
    g = int(rng.integers(0, min(3, nb) + 1))
    w = int(rng.choice([1, 3, 5, 7]))
    r = int(rng.integers(0, 5))
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 3))
    pad = int(rng.integers(0, 3))  # 0 none, 1 prefix lengths, 2 random keys
    return B, H, nb * b, d, b, g, w, r, pad


@pytest.mark.parametrize("seed", range(16))
def test_random_bigbird(seed):
    B, H, n, d, b, g, w, r, pad = _bigbird_params(seed)
    km = None
    if pad == 1:
        km = make_key_mask(B, n, seed=50 + seed)
    elif pad == 2:
        km = make_random_key_mask(B, n, seed=50 + seed, p_valid=0.85)
    bigbird_case(B, H, n, d, b, g, w, r, cfg_id=200 + seed, key_mask=km, seed=seed)


def _longformer_params(seed):
    rng = np.random.default_rng(2000 + seed)
    n = int(rng.integers(200, 2400))
    d = int(rng.choice([64, 128]))
    window = 2 * int(rng.integers(0, 320))
    ng = int(rng.choice([0, 0, 1, 5, 40]))
    H = int(rng.integers(1, 4))
    dil = [int(x) for x in rng.integers(0, 4, size=H)] if rng.random() < 0.6 else None
    causal = bool(rng.random() < 0.4)
    pad = bool(rng.random() < 0.3)
    return n, d, window, ng, H, dil, causal, pad


@pytest.mark.parametrize("seed", range(16))
def test_random_longformer(seed):
    n, d, window, ng, H, dil, causal, pad = _longformer_params(seed)
    gidx = make_global_positions(n, ng, seed=70 + seed) if ng else None
    km = make_key_mask(1, n, seed=80 + seed) if pad else None
    longformer_case(1, H, n, d, window, gidx, cfg_id=300 + seed, key_mask=km, dilation=dil, causal=causal)
