"""The bench's useful-work count against the oracle's explicit masks."""

import numpy as np
import pytest

from block_sparse_long_bigbird_gb300 import accounting
from oracle import bigbird_attended_pairs, bigbird_random_table, longformer_attended_pairs


@pytest.mark.parametrize("n,b,g,w,r", [(4096, 64, 2, 3, 3), (1024, 64, 1, 5, 2), (2048, 128, 2, 3, 3),
                                       (512, 64, 0, 1, 0)])
def test_bigbird_pairs(n, b, g, w, r):
    t = bigbird_random_table(0, 3, n, b, g, w, r)
    assert accounting.bigbird_pairs(n, b, g, w, t) == bigbird_attended_pairs(n, b, g, w, t)
    km = np.zeros((2, n), dtype=np.uint8)
    km[0, : n // 2 + 17] = 1
    km[1, ::5] = 1
    assert accounting.bigbird_pairs(n, b, g, w, t, km) == bigbird_attended_pairs(n, b, g, w, t, km, B=2)


@pytest.mark.parametrize("n,window,G", [(4096, 512, list(range(16))), (1000, 64, [0, 5, 500, 999]),
                                        (512, 0, []), (300, 1000, [3])])
def test_longformer_pairs(n, window, G):
    assert accounting.longformer_pairs(n, window, G) == longformer_attended_pairs(n, window, G)
    km = np.zeros((2, n), dtype=np.uint8)
    km[0, : n // 2 + 3] = 1
    km[1, 1::2] = 1
    assert accounting.longformer_pairs(n, window, G, km) == longformer_attended_pairs(n, window, G, km, B=2)


@pytest.mark.parametrize("n,window,G,dil,causal", [(1000, 64, [0, 5, 500, 999], 1, False),
                                                   (777, 96, [3], 2, True), (512, 128, [], 3, True),
                                                   (300, 1000, [7, 8], 5, False), (640, 32, [0, 1, 2], 0, True)])
def test_longformer_pairs_dilated_causal(n, window, G, dil, causal):
    assert accounting.longformer_pairs(n, window, G, dilation=dil, causal=causal) == \
        longformer_attended_pairs(n, window, G, dilation=[dil], causal=causal)
    km = np.zeros((2, n), dtype=np.uint8)
    km[0, : n // 2 + 3] = 1
    km[1, 1::3] = 1
    assert accounting.longformer_pairs(n, window, G, km, dilation=dil, causal=causal) == \
        longformer_attended_pairs(n, window, G, km, B=2, dilation=[dil], causal=causal)
