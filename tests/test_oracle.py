"""Pins of the float64 oracle to facts fixed outside the oracle itself.

Each test checks the oracle against a published value, a closed form, an
invariant stated by the pages, a special case that reduces to a library
routine (torch's float64 scaled_dot_product_attention on the CPU), or a
scalar brute force written differently from the oracle's vectorised code.
"""

import itertools
import math
import os

import numpy as np
import pytest
import torch

from oracle import (
    bigbird_allowed,
    bigbird_attended_pairs,
    bigbird_random_table,
    longformer_allowed,
    longformer_attended_pairs,
    masked_attention,
    masked_softmax_probs,
    oracle_bigbird,
    oracle_longformer,
    splitmix64_stream,
)
from oracle.attention import bigbird_block_allowed

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _sdpa(q, k, v, mask=None):
    """torch float64 scaled dot-product attention (library routine)."""
    q, k, v = (torch.as_tensor(np.asarray(x, dtype=np.float64)) for x in (q, k, v))
    m = None if mask is None else torch.as_tensor(mask)
    return torch.nn.functional.scaled_dot_product_attention(
        q[None], k[None], v[None], attn_mask=m).numpy()[0]


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- SplitMix64

def test_splitmix64_published_vector():
    lines = [l.split("#")[0].strip() for l in open(os.path.join(GOLDEN, "splitmix64_seed1234567.txt"))]
    lines = [l for l in lines if l]
    seed = int(lines[0].split()[1])
    expected = [int(x) for x in lines[1:]]
    assert splitmix64_stream(seed, len(expected)) == expected


# ------------------------------------------------------------ random table

def _brute_candidates(nb, g, w, j):
    every = set(range(nb))
    glob = set(range(g))
    window = {k for k in every if -(w // 2) <= k - j <= w // 2}
    return every - glob - window


TABLE_CASES = [
    (0, 2, 1024, 64, 2, 3, 3),
    (7, 3, 512, 16, 1, 5, 4),
    (123, 1, 256, 8, 3, 7, 2),
    (99, 2, 128, 16, 0, 1, 2),
    (5, 2, 256, 32, 2, 3, 9),   # fewer candidates than r on some rows
    (11, 1, 192, 64, 1, 3, 3),  # nb = 3: no candidates at all
]


@pytest.mark.parametrize("seed,H,n,b,g,w,r", TABLE_CASES)
def test_random_table_invariants(seed, H, n, b, g, w, r):
    t = bigbird_random_table(seed, H, n, b, g, w, r)
    nb = n // b
    assert t.shape == (H, nb, r) and t.dtype == np.int32
    for h in range(H):
        for j in range(nb):
            row = [int(x) for x in t[h, j]]
            if j < g:
                assert row == [-1] * r, "global rows draw nothing"
                continue
            cand = _brute_candidates(nb, g, w, j)
            k = min(r, len(cand))
            chosen = row[:k]
            assert row[k:] == [-1] * (r - k)
            assert chosen == sorted(chosen)
            assert len(set(chosen)) == k, "distinct"
            assert set(chosen) <= cand, "outside global and window, in range"


def test_random_table_determinism_and_sensitivity():
    a = bigbird_random_table(0, 4, 4096, 64, 2, 3, 3)
    b = bigbird_random_table(0, 4, 4096, 64, 2, 3, 3)
    c = bigbird_random_table(1, 4, 4096, 64, 2, 3, 3)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c)
    for h in range(1, 4):
        assert not np.array_equal(a[0], a[h]), "per-head tables differ"


def test_random_table_sampling_is_uniform():
    # Partial Fisher-Yates picks each candidate with probability k / m.
    nb, g, w, r, j = 12, 1, 3, 3, 6
    m = len(_brute_candidates(nb, g, w, j))
    counts = np.zeros(nb)
    trials = 3000
    for seed in range(trials):
        t = bigbird_random_table(seed, 1, nb * 8, 8, g, w, r)
        for kb in t[0, j]:
            counts[kb] += 1
    cand = sorted(_brute_candidates(nb, g, w, j))
    expect = trials * r / m
    assert counts[[k for k in range(nb) if k not in cand]].sum() == 0
    chi2 = float((((counts[cand] - expect) ** 2) / expect).sum())
    assert chi2 < 30.0, chi2  # 7 degrees of freedom; p < 1e-4 above 30


# ------------------------------------------------------------ BigBird mask

def _brute_bigbird_neigh(nb, g, w, rand_row, qb):
    if qb < g:
        return set(range(nb))
    half = w // 2
    s = set(range(g))
    s |= set(range(max(0, qb - half), min(nb, qb + half + 1)))
    s |= {int(x) for x in rand_row[qb] if x >= 0}
    return s


@pytest.mark.parametrize("seed,H,n,b,g,w,r", TABLE_CASES[:5])
def test_bigbird_mask_matches_enumeration(seed, H, n, b, g, w, r):
    t = bigbird_random_table(seed, H, n, b, g, w, r)
    nb = n // b
    for h in range(H):
        m = bigbird_allowed(n, b, g, w, t[h])
        for i in range(0, n, max(1, b // 3)):
            neigh = _brute_bigbird_neigh(nb, g, w, t[h], i // b)
            expect = np.array([(j // b) in neigh for j in range(n)])
            assert np.array_equal(m[i], expect), (h, i)


def test_bigbird_global_and_window_invariants():
    n, b, g, w, r = 2048, 64, 2, 5, 3
    nb = n // b
    t = bigbird_random_table(3, 1, n, b, g, w, r)
    blk = bigbird_block_allowed(nb, g, w, t[0])
    assert blk[:g].all(), "global blocks attend everything"
    assert blk[:, :g].all(), "everything attends global blocks"
    half = w // 2
    for j in range(g, nb):
        nonrand = blk[j].copy()
        for kb in t[0, j]:
            if kb >= 0:
                nonrand[kb] = False
        nonrand[:g] = False
        idx = np.nonzero(nonrand)[0]
        lo, hi = max(j - half, 0), min(j + half, nb - 1)
        window = [k for k in range(lo, hi + 1) if k >= g]
        assert list(idx) == window, "window is exactly the clipped +-w//2 band"


def test_bigbird_coverage_equals_full_attention():
    # r >= nb: every block is drawn, the pattern is complete -> textbook attention.
    B, H, n, d, b = 1, 2, 256, 16, 32
    t = bigbird_random_table(1, H, n, b, 1, 1, n // b)
    assert bigbird_allowed(n, b, 1, 1, t[0]).all()
    Q, K, V = _rand((B, H, n, d), 1), _rand((B, H, n, d), 2), _rand((B, H, n, d), 3)
    out = oracle_bigbird(Q, K, V, b, 1, 1, t)
    for h in range(H):
        np.testing.assert_allclose(out[0, h], _sdpa(Q[0, h], K[0, h], V[0, h]), rtol=0, atol=1e-12)


def test_bigbird_block_diagonal_equals_per_block_attention():
    # g = 0, w = 1, r = 0: each query block sees only itself (BigBird App. D Eq. 13).
    B, H, n, d, b = 2, 1, 256, 32, 64
    t = bigbird_random_table(0, H, n, b, 0, 1, 0)
    Q, K, V = _rand((B, H, n, d), 4), _rand((B, H, n, d), 5), _rand((B, H, n, d), 6)
    out = oracle_bigbird(Q, K, V, b, 0, 1, t)
    for beta in range(B):
        for j in range(n // b):
            s = slice(j * b, (j + 1) * b)
            ref = _sdpa(Q[beta, 0, s], K[beta, 0, s], V[beta, 0, s])
            np.testing.assert_allclose(out[beta, 0, s], ref, rtol=0, atol=1e-12)


def test_bigbird_matches_sdpa_with_explicit_mask_and_padding():
    # Key padding: padded query rows are exactly 0; the valid region equals
    # library attention on the truncated sequence under the same pattern.
    B, H, n, d, b, g, w, r = 2, 2, 512, 32, 32, 2, 3, 3
    t = bigbird_random_table(9, H, n, b, g, w, r)
    Q, K, V = _rand((B, H, n, d), 7), _rand((B, H, n, d), 8), _rand((B, H, n, d), 9)
    lengths = [301, 512]
    km = np.zeros((B, n), dtype=np.uint8)
    for beta, L in enumerate(lengths):
        km[beta, :L] = 1
    out = oracle_bigbird(Q, K, V, b, g, w, t, key_mask=km)
    for beta, L in enumerate(lengths):
        assert np.all(out[beta, :, L:] == 0.0)
        for h in range(H):
            allowed = bigbird_allowed(n, b, g, w, t[h])[:L, :L]
            ref = _sdpa(Q[beta, h, :L], K[beta, h, :L], V[beta, h, :L], mask=allowed)
            np.testing.assert_allclose(out[beta, h, :L], ref, rtol=0, atol=1e-12)


# ------------------------------------------------------------ Longformer

def test_longformer_mask_invariants():
    n, window = 300, 40
    G = [0, 5, 123, 299]
    m = longformer_allowed(n, window, G)
    for i in range(n):
        for j in range(n):
            expect = (i in G) or (j in G) or abs(i - j) <= window // 2
            assert m[i, j] == expect
    assert m[G].all() and m[:, G].all(), "global attention is symmetric"


def test_longformer_wide_window_equals_full_attention():
    B, H, n, d = 1, 2, 200, 16
    Q, K, V = _rand((B, H, n, d), 10), _rand((B, H, n, d), 11), _rand((B, H, n, d), 12)
    out = oracle_longformer(Q, K, V, 2 * n, [3])
    for h in range(H):
        np.testing.assert_allclose(out[0, h], _sdpa(Q[0, h], K[0, h], V[0, h]), rtol=0, atol=1e-12)


def test_longformer_matches_sdpa_with_band_mask():
    B, H, n, d, window = 1, 1, 384, 32, 64
    G = [0, 1, 200]
    Q, K, V = _rand((B, H, n, d), 13), _rand((B, H, n, d), 14), _rand((B, H, n, d), 15)
    out = oracle_longformer(Q, K, V, window, G)
    i = np.arange(n)
    band = np.abs(i[:, None] - i[None, :]) <= window // 2
    band[G, :] = True
    band[:, G] = True
    np.testing.assert_allclose(out[0, 0], _sdpa(Q[0, 0], K[0, 0], V[0, 0], mask=band), rtol=0, atol=1e-12)


# ------------------------------------------------- Longformer dilation / causal

@pytest.mark.parametrize("dilation,causal", [(0, True), (1, False), (2, True), (3, False)])
def test_longformer_dilated_causal_mask_by_enumeration(dilation, causal):
    # pure-Python enumeration of the window positions i + k (dilation + 1)
    n, window = 70, 8
    G = [4, 33]
    m = longformer_allowed(n, window, G, dilation=dilation, causal=causal)
    for i in range(n):
        seen = set()
        for k in range(-(window // 2), window // 2 + 1):
            j = i + k * (dilation + 1)
            if 0 <= j < n:
                seen.add(j)
        if i in G:
            seen = set(range(n))
        seen |= set(G)
        if causal:
            seen = {j for j in seen if j <= i}
        assert set(np.nonzero(m[i])[0].tolist()) == seen, (i, dilation, causal)


def test_longformer_causal_wide_window_matches_sdpa_is_causal():
    # every previous token in reach: plain causal attention (library routine)
    B, H, n, d = 1, 1, 160, 16
    Q, K, V = _rand((B, H, n, d), 20), _rand((B, H, n, d), 21), _rand((B, H, n, d), 22)
    out = oracle_longformer(Q, K, V, 2 * n, [], causal=True)
    q, k, v = (torch.as_tensor(x[0, 0]) for x in (Q, K, V))
    ref = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], v[None], is_causal=True).numpy()[0]
    np.testing.assert_allclose(out[0, 0], ref, rtol=0, atol=1e-12)


def test_longformer_wide_dilated_window_splits_into_residue_classes():
    # a dilated window reaching every position of its residue class is full
    # attention within each class i mod (dilation + 1), computed here class by class
    B, H, n, d, dil = 1, 2, 150, 16, 2
    Q, K, V = _rand((B, H, n, d), 23), _rand((B, H, n, d), 24), _rand((B, H, n, d), 25)
    out = oracle_longformer(Q, K, V, 2 * n, [], dilation=[dil, dil])
    s = dil + 1
    for h in range(H):
        for r in range(s):
            idx = np.arange(r, n, s)
            ref = _sdpa(Q[0, h, idx], K[0, h, idx], V[0, h, idx])
            np.testing.assert_allclose(out[0, h, idx], ref, rtol=0, atol=1e-12)


def test_longformer_dilated_pair_counts_closed_form():
    # no globals: sum over k in [-w/2, w/2] of the tokens i with 0 <= i + k s < n
    n, window = 64, 8
    for dil, causal in [(1, False), (1, True), (3, False)]:
        s = dil + 1
        ks = range(0, window // 2 + 1) if causal else range(-(window // 2), window // 2 + 1)
        expect = sum(max(0, n - abs(k) * s) for k in ks)
        assert longformer_attended_pairs(n, window, [], dilation=[dil], causal=causal) == expect
    # the numbers for (dilation 1, plain) and (dilation 1, causal), by hand:
    assert longformer_attended_pairs(n, window, [], dilation=[1]) == 536
    assert longformer_attended_pairs(n, window, [], dilation=[1], causal=True) == 300


def test_longformer_causal_globals_only_see_the_past():
    n, window = 50, 4
    G = [10, 30]
    m = longformer_allowed(n, window, G, causal=True)
    assert not np.triu(m, 1).any(), "nothing above the diagonal"
    assert m[30, :31].all() and not m[30, 31:].any()
    assert m[40, 10] and m[40, 30] and not m[5, 10]


# ------------------------------------------------------------ softmax core

def test_softmax_rows_sum_to_one_and_single_key():
    rng = np.random.default_rng(0)
    m, n, d = 40, 70, 16
    q, k, v = rng.standard_normal((m, d)), rng.standard_normal((n, d)), rng.standard_normal((n, d))
    mask = rng.random((m, n)) < 0.3
    mask[0] = False
    p = masked_softmax_probs(q, k, mask)
    sums = p.sum(axis=1)
    assert abs(sums[0]) == 0.0, "a row without keys is all zero"
    assert np.all(np.abs(sums[1:][mask[1:].any(axis=1)] - 1.0) < 1e-12)
    assert np.all(p[~mask] == 0.0)
    single = np.zeros((m, n), dtype=bool)
    pick = rng.integers(0, n, size=m)
    single[np.arange(m), pick] = True
    np.testing.assert_allclose(masked_attention(q, k, v, single), v[pick], rtol=0, atol=0)


def test_scalar_bruteforce_attention():
    # Pure-Python loops with math.exp, written without numpy's vector ops.
    rng = np.random.default_rng(1)
    n, d, b, g, w, r = 24, 4, 4, 1, 3, 1
    t = bigbird_random_table(17, 1, n, b, g, w, r)
    q, k, v = rng.standard_normal((n, d)), rng.standard_normal((n, d)), rng.standard_normal((n, d))
    out = oracle_bigbird(q[None, None], k[None, None], v[None, None], b, g, w, t)[0, 0]
    nb = n // b
    for i in range(n):
        neigh = _brute_bigbird_neigh(nb, g, w, t[0], i // b)
        keys = [j for j in range(n) if j // b in neigh]
        scores = [sum(q[i, c] * k[j, c] for c in range(d)) / math.sqrt(d) for j in keys]
        mx = max(scores)
        ex = [math.exp(s - mx) for s in scores]
        tot = sum(ex)
        ref = [sum(ex[a] * v[keys[a], c] for a in range(len(keys))) / tot for c in range(d)]
        np.testing.assert_allclose(out[i], ref, rtol=0, atol=1e-12)


# ------------------------------------------------------------ work counts

def _golden_counts():
    rows = []
    for line in open(os.path.join(GOLDEN, "pair_counts.txt")):
        line = line.split("#")[0].strip()
        if line:
            rows.append(line.split())
    return rows


@pytest.mark.parametrize("row", _golden_counts(), ids=lambda r: "-".join(r[:2]))
def test_pair_counts_match_closed_form(row):
    if row[0] == "bigbird":
        n, b, g, w, r, expect = map(int, row[1:])
        t = bigbird_random_table(0, 1, n, b, g, w, r)
        assert bigbird_attended_pairs(n, b, g, w, t) == expect
        if n <= 4096:
            assert int(bigbird_allowed(n, b, g, w, t[0]).sum()) == expect
    else:
        n, window, ng, expect = map(int, row[1:])
        assert longformer_attended_pairs(n, window, list(range(ng))) == expect


def test_padded_pair_count_matches_mask():
    n, b, g, w, r = 1024, 64, 2, 3, 3
    t = bigbird_random_table(0, 2, n, b, g, w, r)
    km = np.zeros((2, n), dtype=np.uint8)
    km[0, :700] = 1
    km[1, ::3] = 1
    total = 0
    for h in range(2):
        for beta in range(2):
            valid = km[beta] != 0
            m = bigbird_allowed(n, b, g, w, t[h]) & valid[None, :] & valid[:, None]
            total += int(m.sum())
    assert bigbird_attended_pairs(n, b, g, w, t, key_mask=km, B=2) == total


# ---------------------------------------------------------------------------
# Backward pass: the oracle's gradients against the derivative's definition
# (central finite differences of the pinned forward) and torch autograd.
# ---------------------------------------------------------------------------

def _central_diff_grads(fwd, Q, K, V, dO, eps=1e-5):
    """d(sum(fwd(Q, K, V) * dO)) by central differences, one element at a time."""
    grads = []
    args = [Q.copy(), K.copy(), V.copy()]
    for which in range(3):
        x = args[which]
        g = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            old = x[idx]
            x[idx] = old + eps
            lp = float((fwd(*args) * dO).sum())
            x[idx] = old - eps
            lm = float((fwd(*args) * dO).sum())
            x[idx] = old
            g[idx] = (lp - lm) / (2 * eps)
        grads.append(g)
    return grads


@pytest.mark.parametrize("padded", [False, True])
def test_bigbird_grads_match_finite_differences(padded):
    from oracle import oracle_bigbird_bwd
    n, b, g, w, r, d = 16, 4, 1, 1, 1, 4
    table = bigbird_random_table(3, 1, n, b, g, w, r)
    Q, K, V, dO = (_rand((1, 1, n, d), s) for s in (11, 12, 13, 14))
    km = None
    if padded:
        km = np.ones((1, n), dtype=np.uint8)
        km[0, 13:] = 0
    fwd = lambda q, k, v: oracle_bigbird(q, k, v, b, g, w, table, key_mask=km)
    want = _central_diff_grads(fwd, Q, K, V, dO)
    got = oracle_bigbird_bwd(Q, K, V, dO, b, g, w, table, key_mask=km)
    for gw, gg, name in zip(want, got, "QKV"):
        np.testing.assert_allclose(gg, gw, atol=1e-8, rtol=1e-6, err_msg=f"d{name}")
    if padded:
        assert np.all(got[0][0, 0, 13:] == 0) and np.all(got[1][0, 0, 13:] == 0) and np.all(got[2][0, 0, 13:] == 0)


@pytest.mark.parametrize("dilation,causal,padded", [(0, False, False), (1, True, True), (2, False, True)])
def test_longformer_grads_match_finite_differences(dilation, causal, padded):
    from oracle import oracle_longformer_bwd
    n, window, d = 12, 4, 4
    gidx = np.array([2])
    Q, K, V, dO = (_rand((1, 1, n, d), s) for s in (21, 22, 23, 24))
    km = None
    if padded:
        km = np.ones((1, n), dtype=np.uint8)
        km[0, 10:] = 0
    fwd = lambda q, k, v: oracle_longformer(q, k, v, window, gidx, key_mask=km, dilation=[dilation], causal=causal)
    want = _central_diff_grads(fwd, Q, K, V, dO)
    got = oracle_longformer_bwd(Q, K, V, dO, window, gidx, key_mask=km, dilation=[dilation], causal=causal)
    for gw, gg, name in zip(want, got, "QKV"):
        np.testing.assert_allclose(gg, gw, atol=1e-8, rtol=1e-6, err_msg=f"d{name}")


def _sdpa_grads(q, k, v, mask, dout):
    """torch float64 autograd through scaled_dot_product_attention (library routine)."""
    q, k, v = (torch.tensor(np.asarray(x, dtype=np.float64), requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], v[None],
                                                         attn_mask=torch.as_tensor(mask))[0]
    o.backward(torch.as_tensor(np.asarray(dout, dtype=np.float64)))
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


def test_bigbird_grads_match_torch_autograd():
    from oracle import oracle_bigbird_bwd
    n, b, g, w, r, d, H = 192, 16, 2, 3, 2, 16, 2
    table = bigbird_random_table(5, H, n, b, g, w, r)
    Q, K, V, dO = (_rand((1, H, n, d), s) for s in (31, 32, 33, 34))
    got = oracle_bigbird_bwd(Q, K, V, dO, b, g, w, table, row_chunk=40)
    for h in range(H):
        mask = bigbird_allowed(n, b, g, w, table[h])
        want = _sdpa_grads(Q[0, h], K[0, h], V[0, h], mask, dO[0, h])
        for gw, gg in zip(want, got):
            np.testing.assert_allclose(gg[0, h], gw, atol=1e-12, rtol=1e-9)


@pytest.mark.parametrize("dilation,causal", [(0, False), (3, False), (1, True)])
def test_longformer_grads_match_torch_autograd(dilation, causal):
    from oracle import oracle_longformer_bwd
    n, window, d = 160, 16, 8
    gidx = np.array([0, 1, 77])
    Q, K, V, dO = (_rand((1, 1, n, d), s) for s in (41, 42, 43, 44))
    got = oracle_longformer_bwd(Q, K, V, dO, window, gidx, dilation=[dilation], causal=causal)
    mask = longformer_allowed(n, window, gidx, dilation=dilation, causal=causal)
    want = _sdpa_grads(Q[0, 0], K[0, 0], V[0, 0], mask, dO[0, 0])
    for gw, gg in zip(want, got):
        np.testing.assert_allclose(gg[0, 0], gw, atol=1e-12, rtol=1e-9)


def test_grads_shift_invariance_and_value_sum():
    """Adding one vector c to every key shifts each row's scores by a constant,
    which the softmax ignores, so sum_j dK_j = 0; the rows of P sum to 1 (or are
    0 for a row without keys), so sum_j dV_j = sum of dO over rows with a key."""
    from oracle import oracle_bigbird_bwd
    n, b, g, w, r, d = 256, 32, 1, 3, 2, 8
    table = bigbird_random_table(9, 1, n, b, g, w, r)
    Q, K, V, dO = (_rand((1, 1, n, d), s) for s in (51, 52, 53, 54))
    km = np.ones((1, n), dtype=np.uint8)
    km[0, 200:] = 0
    dQ, dK, dV = oracle_bigbird_bwd(Q, K, V, dO, b, g, w, table, key_mask=km, row_chunk=100)
    np.testing.assert_allclose(dK[0, 0].sum(axis=0), 0.0, atol=1e-12)
    np.testing.assert_allclose(dV[0, 0].sum(axis=0), dO[0, 0, :200].sum(axis=0), atol=1e-12)
    assert np.all(dQ[0, 0, 200:] == 0) and np.all(dK[0, 0, 200:] == 0) and np.all(dV[0, 0, 200:] == 0)


def test_grad_terms_match_scalar_bruteforce():
    """Sum of |term| and sqrt(sum term^2) of every gradient element, from
    scalar loops over the definitions (softmax, dS, then the products)."""
    from oracle import masked_attention_grad_terms
    m, n, d = 5, 6, 3
    rng = np.random.default_rng(61)
    q, k, v, do = rng.standard_normal((m, d)), rng.standard_normal((n, d)), rng.standard_normal((n, d)), \
        rng.standard_normal((m, d))
    mask = rng.random((m, n)) < 0.6
    mask[0, :] = False  # a row without keys
    sc = 1.0 / math.sqrt(d)
    P = np.zeros((m, n))
    dS = np.zeros((m, n))
    for i in range(m):
        keys = [j for j in range(n) if mask[i, j]]
        if not keys:
            continue
        s = {j: sc * sum(q[i, c] * k[j, c] for c in range(d)) for j in keys}
        mx = max(s.values())
        z = sum(math.exp(s[j] - mx) for j in keys)
        for j in keys:
            P[i, j] = math.exp(s[j] - mx) / z
        dp = {j: sum(do[i, c] * v[j, c] for c in range(d)) for j in keys}
        Di = sum(P[i, j] * dp[j] for j in keys)
        for j in keys:
            dS[i, j] = P[i, j] * (dp[j] - Di)
    (qa, qr), (ka, kr), (va, vr) = masked_attention_grad_terms(q, k, v, mask, do)
    for i in range(m):
        for c in range(d):
            t = [sc * dS[i, j] * k[j, c] for j in range(n)]
            assert math.isclose(qa[i, c], sum(abs(x) for x in t), rel_tol=1e-12, abs_tol=1e-15)
            assert math.isclose(qr[i, c], math.sqrt(sum(x * x for x in t)), rel_tol=1e-12, abs_tol=1e-15)
    for j in range(n):
        for c in range(d):
            t = [sc * dS[i, j] * q[i, c] for i in range(m)]
            u = [P[i, j] * do[i, c] for i in range(m)]
            assert math.isclose(ka[j, c], sum(abs(x) for x in t), rel_tol=1e-12, abs_tol=1e-15)
            assert math.isclose(kr[j, c], math.sqrt(sum(x * x for x in t)), rel_tol=1e-12, abs_tol=1e-15)
            assert math.isclose(va[j, c], sum(abs(x) for x in u), rel_tol=1e-12, abs_tol=1e-15)
            assert math.isclose(vr[j, c], math.sqrt(sum(x * x for x in u)), rel_tol=1e-12, abs_tol=1e-15)


def test_bf16_rounded_factors_stay_inside_the_term_bound():
    """Rounding P and dS to bf16 (a relative error of at most 2^-9 each)
    moves every gradient element by at most 2^-9 * sum |term|."""
    from oracle import masked_attention_grad_terms
    n, d = 512, 64
    rng = np.random.default_rng(62)
    q, k, v, do = (rng.standard_normal((n, d)) for _ in range(4))
    mask = bigbird_allowed(n, 64, 1, 3, bigbird_random_table(1, 1, n, 64, 1, 3, 2)[0])
    sc = 1.0 / math.sqrt(d)
    P = masked_softmax_probs(q, k, mask)
    dp = do @ v.T
    dS = P * (dp - (P * dp).sum(axis=1)[:, None])
    to_bf16 = lambda x: torch.as_tensor(x).to(torch.bfloat16).to(torch.float64).numpy()
    Pb, dSb = to_bf16(P), to_bf16(dS)
    (qa, _), (ka, _), (va, _) = masked_attention_grad_terms(q, k, v, mask, do)
    assert np.all(np.abs(sc * (dSb - dS) @ k) <= 2.0 ** -9 * qa + 1e-15)
    assert np.all(np.abs(sc * (dSb - dS).T @ q) <= 2.0 ** -9 * ka + 1e-15)
    assert np.all(np.abs((Pb - P).T @ do) <= 2.0 ** -9 * va + 1e-15)


# ---------------------------------------------------------------------------
# Longformer separate projections for global attention (Sec. 3.1)
# ---------------------------------------------------------------------------

def test_longformer_global_projections_split_rows():
    """Global rows equal full softmax attention of (Qg, Kg, Vg) over the keys
    they see (torch SDPA); the other rows equal the single-projection oracle
    and ignore Qg, Kg, Vg."""
    n, window, d = 200, 16, 8
    gidx = np.array([0, 3, 150])
    Q, K, V, Qg, Kg, Vg = (_rand((1, 1, n, d), s) for s in (71, 72, 73, 74, 75, 76))
    for causal in (False, True):
        got = oracle_longformer(Q, K, V, window, gidx, causal=causal, Qg=Qg, Kg=Kg, Vg=Vg)[0, 0]
        plain = oracle_longformer(Q, K, V, window, gidx, causal=causal)[0, 0]
        other = np.setdiff1d(np.arange(n), gidx)
        np.testing.assert_allclose(got[other], plain[other], rtol=0, atol=0)
        mask = longformer_allowed(n, window, gidx, causal=causal)
        want = _sdpa(Qg[0, 0, gidx], Kg[0, 0], Vg[0, 0], mask[gidx])
        np.testing.assert_allclose(got[gidx], want, atol=1e-12, rtol=1e-10)
    # the same tensors as both sets give the plain oracle
    same = oracle_longformer(Q, K, V, window, gidx, Qg=Q, Kg=K, Vg=V)
    np.testing.assert_allclose(same, oracle_longformer(Q, K, V, window, gidx), rtol=0, atol=0)


# ---------------------------------------------------------------------------
# BigBird-ETC (added global tokens, no random blocks)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n,g,b,w", [(40, 5, 4, 3), (64, 8, 8, 1), (50, 0, 5, 3), (37, 3, 4, 5)])
def test_etc_mask_matches_enumeration(n, g, b, w):
    from oracle import bigbird_etc_allowed
    got = bigbird_etc_allowed(n, g, b, w)
    for i in range(n):
        for j in range(n):
            if i < g or j < g:
                want = True
            else:
                want = abs((i - g) // b - (j - g) // b) <= w // 2
            assert got[i, j] == want, (i, j)


def test_etc_equals_itc_layout_with_block_aligned_globals():
    """With b dividing g, ETC over n tokens is ITC with g/b global blocks and no random blocks."""
    from oracle import bigbird_etc_allowed
    n, g, b, w = 640, 128, 64, 3
    itc = bigbird_allowed(n, b, g // b, w, np.full((n // b, 0), -1))
    np.testing.assert_array_equal(bigbird_etc_allowed(n, g, b, w), itc)


def test_etc_padded_prefix_equals_unpadded():
    """g not a multiple of b: pad the global prefix to a whole block with tokens
    that key padding removes; the real rows are unchanged."""
    from oracle import oracle_bigbird_etc
    g, b, w, nreg, d = 23, 16, 3, 96, 8
    gp = -(-g // b) * b
    Q, K, V = (_rand((1, 1, g + nreg, d), s) for s in (81, 82, 83))
    ref = oracle_bigbird_etc(Q, K, V, g, b, w)
    pad = lambda x: np.concatenate([x[:, :, :g], np.zeros((1, 1, gp - g, d)), x[:, :, g:]], axis=2)
    km = np.ones((1, gp + nreg), dtype=np.uint8)
    km[0, g:gp] = 0
    got = oracle_bigbird_etc(pad(Q), pad(K), pad(V), gp, b, w, key_mask=km)
    keep = np.concatenate([np.arange(g), np.arange(gp, gp + nreg)])
    np.testing.assert_allclose(got[0, 0, keep], ref[0, 0], atol=1e-12, rtol=1e-12)
    assert np.all(got[0, 0, g:gp] == 0)


def test_longformer_global_projection_grads_match_finite_differences():
    """The six gradients of the separate-projection forward, by central differences."""
    from oracle import oracle_longformer_bwd
    n, window, d = 12, 4, 3
    gidx = np.array([2, 9])
    X = [_rand((1, 1, n, d), s) for s in (101, 102, 103, 104, 105, 106)]
    dO = _rand((1, 1, n, d), 107)
    km = np.ones((1, n), dtype=np.uint8)
    km[0, 11] = 0
    for causal in (False, True):
        fwd = lambda q, k, v, qg, kg, vg: oracle_longformer(q, k, v, window, gidx, key_mask=km, causal=causal,
                                                           Qg=qg, Kg=kg, Vg=vg)
        got = oracle_longformer_bwd(*X[:3], dO, window, gidx, key_mask=km, causal=causal,
                                    Qg=X[3], Kg=X[4], Vg=X[5])
        eps = 1e-5
        for which in range(6):
            x = X[which]
            want = np.zeros_like(x)
            for idx in np.ndindex(*x.shape):
                old = x[idx]
                x[idx] = old + eps
                lp = float((fwd(*X) * dO).sum())
                x[idx] = old - eps
                lm = float((fwd(*X) * dO).sum())
                x[idx] = old
                want[idx] = (lp - lm) / (2 * eps)
            np.testing.assert_allclose(got[which], want, atol=1e-8, rtol=1e-6, err_msg=f"grad {which} causal={causal}")


def test_sampled_backward_equals_full_backward():
    """The sampled backward (for long sequences) reproduces the full backward's
    dQ rows and dK, dV key blocks, term sizes included."""
    from oracle import oracle_bigbird_bwd, oracle_bigbird_bwd_sampled
    n, b, g, w, r, d = 512, 32, 2, 3, 2, 8
    table = bigbird_random_table(4, 1, n, b, g, w, r)
    Q, K, V, dO = (_rand((1, 1, n, d), s) for s in (121, 122, 123, 124))
    km = np.ones((1, n), dtype=np.uint8)
    km[0, 470:] = 0
    full, terms = oracle_bigbird_bwd(Q, K, V, dO, b, g, w, table, key_mask=km, terms=True)
    rows = np.array([0, 5, 100, 101, 300, 511])
    kblocks = [3, 7, 15]
    keys = np.concatenate([np.arange(k * b, (k + 1) * b) for k in kblocks])
    (dq, tq), (dk, tk), (dv, tv) = oracle_bigbird_bwd_sampled(Q[0, 0], K[0, 0], V[0, 0], dO[0, 0], b, g, w,
                                                              table[0], rows, kblocks, key_valid=km[0], row_chunk=50)
    np.testing.assert_allclose(dq, full[0][0, 0, rows], atol=1e-12)
    np.testing.assert_allclose(dk, full[1][0, 0, keys], atol=1e-12)
    np.testing.assert_allclose(dv, full[2][0, 0, keys], atol=1e-12)
    for got, want, idx in ((tq, terms[0], rows), (tk, terms[1], keys), (tv, terms[2], keys)):
        np.testing.assert_allclose(got[0], want[0][0, 0, idx], atol=1e-12)
        np.testing.assert_allclose(got[1], want[1][0, 0, idx], atol=1e-12)
