"""Useful-work accounting for the sparse-attention forward and backward.

Useful FLOPs = 4 * d per attended pair (a valid query and an allowed valid
key): 2 d for the score Q_i . K_j and 2 d for accumulating P_ij V_j. The
backward counts 10 * d per pair: the five products a backward needs (the
score recomputed, dP_ij = dO_i . V_j, and the accumulations of dV, dQ and dK),
whatever extra work an implementation does. The pair
count follows the patterns' definitions ("Big Bird" Sec. 2 / App. D;
"Longformer" Sec. 3.1) at block granularity for BigBird and row by row for
Longformer; it is host-side bookkeeping and never enters a kernel.
"""

import numpy as np

FWD_FLOPS_PER_PAIR_PER_D = 4
BWD_FLOPS_PER_PAIR_PER_D = 10


def bigbird_block_sets(nb, g, w, rand_row):
    """Sorted key-block list of every query block of one head."""
    half = w // 2
    sets = []
    for j in range(nb):
        if j < g:
            sets.append(np.arange(nb))
            continue
        s = set(range(min(g, nb)))
        s.update(range(max(0, j - half), min(nb, j + half + 1)))
        s.update(int(x) for x in rand_row[j] if 0 <= x < nb)
        sets.append(np.array(sorted(s)))
    return sets


def bigbird_pairs(n, b, g, w, table, key_mask=None):
    """Attended pairs summed over batch entries and heads.

    table: int [H, n // b, r]; key_mask: uint8/bool [B, n] or None (then B = 1
    and the caller multiplies by the batch size).
    """
    table = np.asarray(table)
    H, nb = table.shape[0], n // b
    masks = [None] if key_mask is None else [np.asarray(m) != 0 for m in key_mask]
    total = 0
    for h in range(H):
        sets = bigbird_block_sets(nb, g, w, table[h])
        for valid in masks:
            if valid is None:
                total += sum(len(s) for s in sets) * b * b
            else:
                per_blk = valid.reshape(nb, b).sum(axis=1).astype(np.int64)
                total += int(sum(per_blk[j] * per_blk[s].sum() for j, s in enumerate(sets)))
    return total


def longformer_pairs(n, window, global_idx, key_mask=None, dilation=0, causal=False):
    """Attended pairs of one head summed over batch entries (B = 1 if no mask).

    ``dilation``: the head's window gaps (stride dilation + 1); ``causal``: no
    key after the query ("Longformer", Sec. 3.1 and App. B). Counted per row
    with prefix sums over each residue class of the stride.
    """
    half = window // 2
    s = int(dilation) + 1
    reach = half * s
    G = np.unique(np.asarray(global_idx, dtype=np.int64))
    is_g = np.zeros(n, dtype=bool)
    is_g[G] = True
    masks = [np.ones(n, dtype=bool)] if key_mask is None else [np.asarray(m) != 0 for m in key_mask]
    i = np.arange(n)
    m = -(-n // s)  # positions per residue class (the last classes may hold one fewer)
    total = 0
    for valid in masks:
        # per residue class c: prefix counts of valid keys and of valid global keys
        vc = np.zeros((s, m + 1), dtype=np.int64)
        gc = np.zeros((s, m + 1), dtype=np.int64)
        for c in range(s):
            pos = np.arange(c, n, s)
            vc[c, 1:len(pos) + 1] = np.cumsum(valid[pos])
            vc[c, len(pos) + 1:] = vc[c, len(pos)]
            gc[c, 1:len(pos) + 1] = np.cumsum(valid[pos] & is_g[pos])
            gc[c, len(pos) + 1:] = gc[c, len(pos)]
        c = i % s
        lo = i - np.minimum(reach, (i // s) * s)          # first band position of the class
        hi_full = i + np.minimum(reach, ((n - 1 - i) // s) * s)
        hi = i if causal else hi_full
        band = vc[c, hi // s + 1] - vc[c, lo // s]
        band_g = gc[c, hi // s + 1] - gc[c, lo // s]
        cum_v = np.concatenate([[0], np.cumsum(valid)])
        cum_g = np.concatenate([[0], np.cumsum(valid & is_g)])
        upto = (i + 1) if causal else np.full(n, n)
        glob_keys = cum_g[upto]                       # valid global keys the row may see
        row_counts = np.where(is_g, cum_v[upto], band + glob_keys - band_g)
        total += int(row_counts[valid].sum())
    return total
