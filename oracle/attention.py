"""Masked dense softmax attention in float64: the oracle's definition of the
BigBird and Longformer forward passes (test infrastructure, CPU only).

What is computed (per batch entry beta and head h):

    S       = Q K^T / sqrt(d)                                  (Longformer Sec. 3.1, Eq. 1)
    M[i, j] = allowed(i, j) and valid(j) and valid(i)          (BigBird Sec. 2, Eq. AT: the
                                                                neighbourhood N(i) of graph D)
    P[i, :] = softmax of S[i, :] over {j : M[i, j]}
    O[i, :] = sum_j P[i, j] V[j, :]   if row i has an allowed key, else 0

No blocking, no fusion, no reordering: the explicit n x n (or rows x n) boolean
mask is built from the pattern's definition and applied to the dense score
matrix. BigBird App. D (Fig. 6 caption) states that its blockified product
yields exactly the sparse matrix of its Fig. 3(d); a faster implementation must
therefore equal this masked dense computation up to rounding.

Readings where the pages are silent or garbled (all recorded in the design notes):
  * BigBird global blocks are blocks 0..g-1 (ITC: existing tokens made global,
    blog Sec. 2.3 "e.g. the first 128 tokens"); g, w, r are counted in blocks.
  * The BigBird window reaches w // 2 blocks each side and is clipped at the
    sequence ends (no circular wrap); Longformer reaches window // 2 tokens each
    side, also clipped.
  * Key padding (valid = key_mask) removes keys; padded query rows are zero.
  * A row with no allowed valid key outputs zeros.
"""

import math

import numpy as np


# ---------------------------------------------------------------------------
# Attention patterns (boolean "allowed" masks)
# ---------------------------------------------------------------------------

def bigbird_block_allowed(nb, g, w, rand_row):
    """Block-level neighbourhood of BigBird-ITC, bool [nb, nb].

    ``rand_row`` is one head's random table [nb, r] (-1 = no block). Query block
    qb attends key block kb when (BigBird Sec. 2 / blog Sec. 2.1-2.3):
      * qb is a global block (qb < g): global tokens attend everything;
      * kb is a global block (kb < g): everything attends global tokens;
      * |qb - kb| <= w // 2: the sliding window of w blocks;
      * kb is one of qb's random blocks.
    """
    half = w // 2
    allowed = np.zeros((nb, nb), dtype=bool)
    for qb in range(nb):
        randoms = set(int(x) for x in rand_row[qb] if x >= 0)
        for kb in range(nb):
            if qb < g:
                allowed[qb, kb] = True
            elif kb < g:
                allowed[qb, kb] = True
            elif abs(qb - kb) <= half:
                allowed[qb, kb] = True
            elif kb in randoms:
                allowed[qb, kb] = True
    return allowed


def bigbird_allowed(n, b, g, w, rand_row, rows=None):
    """Token-level BigBird mask, bool [len(rows), n]: token i sees token j iff
    block i // b sees block j // b (blockified pattern, BigBird App. D)."""
    nb = n // b
    blk = bigbird_block_allowed(nb, g, w, rand_row)
    rows = np.arange(n) if rows is None else np.asarray(rows)
    cols = np.arange(n)
    return blk[rows[:, None] // b, cols[None, :] // b]


def longformer_allowed(n, window, global_idx, rows=None, dilation=0, causal=False):
    """Longformer mask, bool [len(rows), n] (Longformer Sec. 3.1).

    Token i sees token j when i or j carries global attention (symmetric: a
    global token attends all tokens and all tokens attend it), or when j lies in
    i's sliding window: window // 2 positions on each side, clipped at the ends.
    Dilated sliding window (Sec. 3.1, Fig. 2(c)): the window has gaps of size
    `dilation` between attended positions, so the positions are i + k (dilation
    + 1) for |k| <= window // 2 (dilation 0 is the plain window, as in Tab. 12).
    Autoregressive mode (App. B: each token attends to previous tokens only):
    with `causal`, nothing with j > i is allowed, global tokens included.
    """
    rows = np.arange(n) if rows is None else np.asarray(rows)
    cols = np.arange(n)
    is_global = np.zeros(n, dtype=bool)
    is_global[np.asarray(global_idx, dtype=np.int64)] = True
    stride = int(dilation) + 1
    diff = rows[:, None] - cols[None, :]  # i - j
    band = (np.abs(diff) <= (window // 2) * stride) & (diff % stride == 0)
    allowed = band | is_global[rows][:, None] | is_global[None, :]
    if causal:
        allowed &= diff >= 0
    return allowed


def bigbird_etc_allowed(n, g_tokens, b, w, rows=None):
    """BigBird-ETC mask, bool [len(rows), n] ("Big Bird", Sec. 2 global tokens,
    extended construction; App. E Tab. 8 and the QA tables: g added global
    tokens, window w blocks, no random blocks).

    The sequence holds the g_tokens added global tokens first, then the regular
    tokens. A global token sees every token and every token sees it. A regular
    token at position p sees the regular tokens whose block (p - g_tokens) // b
    is within w // 2 of its own, clipped at the ends.
    """
    rows = np.arange(n) if rows is None else np.asarray(rows)
    cols = np.arange(n)
    gi = rows < g_tokens
    gj = cols < g_tokens
    bi = (rows - g_tokens) // b
    bj = (cols - g_tokens) // b
    window = (np.abs(bi[:, None] - bj[None, :]) <= w // 2) & ~gi[:, None] & ~gj[None, :]
    return window | gi[:, None] | gj[None, :]


def oracle_bigbird_etc(Q, K, V, g_tokens, b, w, key_mask=None, rows=None):
    """BigBird-ETC attention forward, float64 [B, H, len(rows), d]."""
    Q, K, V = _as_f64(Q), _as_f64(K), _as_f64(V)
    B, H, n, d = Q.shape
    rows = np.arange(n) if rows is None else np.asarray(rows)
    out = np.zeros((B, H, len(rows), d), dtype=np.float64)
    mask0 = bigbird_etc_allowed(n, g_tokens, b, w, rows)
    for beta in range(B):
        kv = None if key_mask is None else np.asarray(key_mask[beta]) != 0
        mask = _apply_validity(mask0, rows, kv)
        for h in range(H):
            out[beta, h] = masked_attention(Q[beta, h, rows], K[beta, h], V[beta, h], mask)
    return out


# ---------------------------------------------------------------------------
# Masked softmax attention
# ---------------------------------------------------------------------------

def masked_softmax_probs(q, k, mask):
    """P = softmax over the allowed keys of (q k^T / sqrt(d)), float64.

    q: [m, d], k: [n, d], mask: bool [m, n]. Rows without an allowed key are 0.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    d = q.shape[1]
    s = (q @ k.T) / math.sqrt(d)
    s = np.where(mask, s, -np.inf)
    any_allowed = mask.any(axis=1)
    row_max = np.where(any_allowed, s.max(axis=1, initial=-np.inf), 0.0)
    e = np.where(mask, np.exp(s - row_max[:, None]), 0.0)
    denom = e.sum(axis=1)
    denom = np.where(any_allowed, denom, 1.0)
    return e / denom[:, None]


def masked_attention(q, k, v, mask):
    """O = P V for P = masked_softmax_probs(q, k, mask); float64 [m, d]."""
    p = masked_softmax_probs(q, k, mask)
    return p @ np.asarray(v, dtype=np.float64)


def _apply_validity(mask, rows, key_valid):
    if key_valid is None:
        return mask
    key_valid = np.asarray(key_valid, dtype=bool)
    return mask & key_valid[None, :] & key_valid[rows][:, None]


def _as_f64(x):
    """Upcast exactly to float64 (accepts numpy arrays or CPU torch tensors)."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def oracle_bigbird(Q, K, V, b, g, w, rand_table, key_mask=None, rows=None,
                   row_chunk=1024):
    """BigBird-ITC attention forward, float64 [B, H, len(rows), d].

    Q, K, V: [B, H, n, d] (any float type; upcast exactly). rand_table:
    int [H, n // b, r], shared by all batch entries. key_mask: [B, n], nonzero =
    valid token, or None. rows: query rows to compute (default all).
    """
    Q, K, V = _as_f64(Q), _as_f64(K), _as_f64(V)
    rand_table = np.asarray(rand_table)
    B, H, n, d = Q.shape
    rows = np.arange(n) if rows is None else np.asarray(rows)
    out = np.zeros((B, H, len(rows), d), dtype=np.float64)
    for h in range(H):
        blk = bigbird_block_allowed(n // b, g, w, rand_table[h])
        for beta in range(B):
            kv = None if key_mask is None else np.asarray(key_mask[beta]) != 0
            for c0 in range(0, len(rows), row_chunk):
                rr = rows[c0:c0 + row_chunk]
                mask = blk[rr[:, None] // b, np.arange(n)[None, :] // b]
                mask = _apply_validity(mask, rr, kv)
                out[beta, h, c0:c0 + len(rr)] = masked_attention(
                    Q[beta, h, rr], K[beta, h], V[beta, h], mask)
    return out


def oracle_longformer(Q, K, V, window, global_idx, key_mask=None, rows=None,
                      row_chunk=1024, dilation=None, causal=False, Qg=None, Kg=None, Vg=None):
    """Longformer sliding-window + global attention forward, float64.

    ``dilation``: per-head dilation [H] (None: 0 for every head); ``causal``:
    autoregressive mode. See ``longformer_allowed``.

    Separate projections for global attention (Longformer Sec. 3.1, "Linear
    Projections for Global Attention"): with ``Qg``, ``Kg``, ``Vg`` given
    ([B, H, n, d] each), the row of a global token is computed from Qg against
    Kg and Vg over every key it may see, and every other row from Q, K, V as
    usual (including its scores against global keys). Without them the global
    rows use Q, K, V.
    """
    Q, K, V = _as_f64(Q), _as_f64(K), _as_f64(V)
    sep = Qg is not None
    if sep:
        Qg, Kg, Vg = _as_f64(Qg), _as_f64(Kg), _as_f64(Vg)
    B, H, n, d = Q.shape
    dil = np.zeros(H, dtype=np.int64) if dilation is None else np.asarray(dilation, dtype=np.int64)
    rows = np.arange(n) if rows is None else np.asarray(rows)
    is_global = np.zeros(n, dtype=bool)
    is_global[np.asarray(global_idx, dtype=np.int64)] = True
    out = np.zeros((B, H, len(rows), d), dtype=np.float64)
    for beta in range(B):
        kv = None if key_mask is None else np.asarray(key_mask[beta]) != 0
        for c0 in range(0, len(rows), row_chunk):
            rr = rows[c0:c0 + row_chunk]
            masks = {}
            for h in range(H):
                if dil[h] not in masks:
                    masks[dil[h]] = _apply_validity(
                        longformer_allowed(n, window, global_idx, rr, dilation=dil[h], causal=causal), rr, kv)
                mask = masks[dil[h]]
                o = masked_attention(Q[beta, h, rr], K[beta, h], V[beta, h], mask)
                if sep:
                    g = is_global[rr]
                    if g.any():
                        o[g] = masked_attention(Qg[beta, h, rr[g]], Kg[beta, h], Vg[beta, h], mask[g])
                out[beta, h, c0:c0 + len(rr)] = o
    return out


# ---------------------------------------------------------------------------
# Backward pass: gradients of the forward above
# ---------------------------------------------------------------------------
#
# The pages train every model through this attention (BigBird App. E.1, MLM
# pretraining; Longformer Sec. 5, continued MLM pretraining with gradient
# updates) but print no backward formulas: the backward is the exact
# derivative of the forward definition. For a loss L with upstream gradient
# dO = dL/dO and the row-wise masked softmax P of the forward:
#
#     dV      = P^T dO                      (O = P V is linear in V)
#     dP      = dO V^T
#     D_i     = sum_j P_ij dP_ij            (= dO_i . O_i)
#     dS_ij   = P_ij (dP_ij - D_i)          (softmax Jacobian on the allowed keys;
#                                            P_ij = 0 off the mask, so dS_ij = 0 there)
#     dQ      = dS K / sqrt(d),  dK = dS^T Q / sqrt(d)
#
# Rows without an allowed key (padded queries) have P_i = 0, hence zero
# gradient, matching their constant zero output.

def masked_attention_grads(q, k, v, mask, dout):
    """(dq, dk, dv) of O = masked_attention(q, k, v, mask) for dL/dO = dout, float64.

    q, dout: [m, d]; k, v: [n, d]; mask: bool [m, n].
    """
    q, k, v, dout = (_as_f64(x) for x in (q, k, v, dout))
    scale = 1.0 / math.sqrt(q.shape[1])
    p = masked_softmax_probs(q, k, mask)
    dv = p.T @ dout
    dp = dout @ v.T
    rowdot = (p * dp).sum(axis=1)
    ds = p * (dp - rowdot[:, None])
    return scale * (ds @ k), scale * (ds.T @ q), dv


def masked_attention_grad_terms(q, k, v, mask, dout):
    """Size of the sums behind each gradient element, for error analysis.

    Every element of dQ, dK and dV is a sum of products (dQ_ic = sum_j t_j with
    t_j = dS_ij K_jc / sqrt(d), dK_jc over i of dS_ij Q_ic / sqrt(d), dV_jc
    over i of P_ij dO_ic). Returns, for (dq, dk, dv) in turn, the pair
    (sum_t |t|, sqrt(sum_t t^2)): the first bounds the effect of rounding every
    factor P or dS by a relative e (at most e * sum |t|), the second is the
    scale of that effect when the roundings are independent.
    """
    q, k, v, dout = (_as_f64(x) for x in (q, k, v, dout))
    scale = 1.0 / math.sqrt(q.shape[1])
    p = masked_softmax_probs(q, k, mask)
    dp = dout @ v.T
    ds = p * (dp - (p * dp).sum(axis=1)[:, None])
    a, a2 = np.abs(ds), ds * ds
    return ((scale * (a @ np.abs(k)), scale * np.sqrt(a2 @ (k * k))),
            (scale * (a.T @ np.abs(q)), scale * np.sqrt(a2.T @ (q * q))),
            (p.T @ np.abs(dout), np.sqrt((p * p).T @ (dout * dout))))


def _grads_over_rows(Qh, Kh, Vh, dOh, mask_of_rows, n, row_chunk, terms=False):
    """Sum the per-row contributions to dK and dV over row chunks of one head
    (dQ rows are independent); the chunks only bound memory. With ``terms``,
    also return the term sizes of ``masked_attention_grad_terms`` (the squared
    sums add over chunks)."""
    dQ = np.zeros_like(Qh)
    dK = np.zeros_like(Kh)
    dV = np.zeros_like(Vh)
    tq = [np.zeros_like(Qh), np.zeros_like(Qh)]
    tk = [np.zeros_like(Kh), np.zeros_like(Kh)]
    tv = [np.zeros_like(Vh), np.zeros_like(Vh)]
    for c0 in range(0, n, row_chunk):
        rr = np.arange(c0, min(n, c0 + row_chunk))
        mask = mask_of_rows(rr)
        dq, dk, dv = masked_attention_grads(Qh[rr], Kh, Vh, mask, dOh[rr])
        dQ[rr] = dq
        dK += dk
        dV += dv
        if terms:
            (qa, qr), (ka, kr), (va, vr) = masked_attention_grad_terms(Qh[rr], Kh, Vh, mask, dOh[rr])
            tq[0][rr], tq[1][rr] = qa, qr
            tk[0] += ka
            tk[1] += kr * kr
            tv[0] += va
            tv[1] += vr * vr
    if not terms:
        return dQ, dK, dV
    tk[1], tv[1] = np.sqrt(tk[1]), np.sqrt(tv[1])
    return (dQ, dK, dV), (tuple(tq), tuple(tk), tuple(tv))


def oracle_bigbird_bwd(Q, K, V, dO, b, g, w, rand_table, key_mask=None, row_chunk=1024, terms=False):
    """Gradients (dQ, dK, dV), float64 [B, H, n, d], of the BigBird-ITC forward
    ``oracle_bigbird`` for the upstream gradient dO [B, H, n, d]. With
    ``terms``, returns ((dQ, dK, dV), term sizes), the term sizes as in
    ``masked_attention_grad_terms`` with a leading [B, H]."""
    Q, K, V, dO = _as_f64(Q), _as_f64(K), _as_f64(V), _as_f64(dO)
    rand_table = np.asarray(rand_table)
    B, H, n, d = Q.shape
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    T = [[np.zeros_like(Q), np.zeros_like(Q)] for _ in range(3)] if terms else None
    for h in range(H):
        blk = bigbird_block_allowed(n // b, g, w, rand_table[h])
        for beta in range(B):
            kv = None if key_mask is None else np.asarray(key_mask[beta]) != 0

            def mask_of_rows(rr):
                return _apply_validity(blk[rr[:, None] // b, np.arange(n)[None, :] // b], rr, kv)

            res = _grads_over_rows(Q[beta, h], K[beta, h], V[beta, h], dO[beta, h], mask_of_rows, n,
                                   row_chunk, terms)
            if terms:
                res, tt = res
                for which in range(3):
                    for kind in range(2):
                        T[which][kind][beta, h] = tt[which][kind]
            dQ[beta, h], dK[beta, h], dV[beta, h] = res
    return ((dQ, dK, dV), T) if terms else (dQ, dK, dV)


def oracle_bigbird_bwd_sampled(Qh, Kh, Vh, dOh, b, g, w, rand_row, rows, key_blocks, key_valid=None,
                               row_chunk=512):
    """Exact gradients of one head at sampled places, for sequences too long for
    ``oracle_bigbird_bwd``: dQ on ``rows``, and dK, dV on the keys of
    ``key_blocks``, with the term sizes of ``masked_attention_grad_terms``.

    dQ_i needs only row i's own neighbourhood. dK_j and dV_j sum over the rows
    that see key j; for the sampled key blocks those rows are found from the
    block mask (its transpose), so every contribution is included.
    Returns ((dq, (A, R)), (dk, (A, R)), (dv, (A, R))): dq [len(rows), d],
    dk and dv [len(keys), d] in the order of the sampled blocks' keys.
    """
    Qh, Kh, Vh, dOh = (_as_f64(x) for x in (Qh, Kh, Vh, dOh))
    n, d = Qh.shape
    nb = n // b
    blk = bigbird_block_allowed(nb, g, w, rand_row)
    kv = None if key_valid is None else np.asarray(key_valid, dtype=bool)
    cols = np.arange(n)

    def mask_of(rr):
        return _apply_validity(blk[rr[:, None] // b, cols[None, :] // b], rr, kv)

    rows = np.asarray(rows)
    dq = np.zeros((len(rows), d))
    qa = np.zeros((len(rows), d))
    qr = np.zeros((len(rows), d))
    for c0 in range(0, len(rows), row_chunk):
        rr = rows[c0:c0 + row_chunk]
        args = (Qh[rr], Kh, Vh, mask_of(rr), dOh[rr])
        dq[c0:c0 + len(rr)] = masked_attention_grads(*args)[0]
        (a, r2), _, _ = masked_attention_grad_terms(*args)
        qa[c0:c0 + len(rr)], qr[c0:c0 + len(rr)] = a, r2
    keys = np.concatenate([np.arange(kb * b, (kb + 1) * b) for kb in key_blocks])
    seeing = np.nonzero(blk[:, np.asarray(key_blocks)].any(axis=1))[0]  # query blocks that see a sampled block
    srows = np.concatenate([np.arange(qb * b, (qb + 1) * b) for qb in seeing])
    dk = np.zeros((n, d))
    dv = np.zeros((n, d))
    ka, kr2, va, vr2 = (np.zeros((n, d)) for _ in range(4))
    for c0 in range(0, len(srows), row_chunk):
        rr = srows[c0:c0 + row_chunk]
        args = (Qh[rr], Kh, Vh, mask_of(rr), dOh[rr])
        _, k1, v1 = masked_attention_grads(*args)
        _, (a1, r1), (a2, r2) = masked_attention_grad_terms(*args)
        dk += k1
        dv += v1
        ka += a1
        kr2 += r1 * r1
        va += a2
        vr2 += r2 * r2
    return ((dq, (qa, qr)), (dk[keys], (ka[keys], np.sqrt(kr2[keys]))),
            (dv[keys], (va[keys], np.sqrt(vr2[keys]))))


def oracle_longformer_bwd(Q, K, V, dO, window, global_idx, key_mask=None, dilation=None,
                          causal=False, row_chunk=1024, terms=False, Qg=None, Kg=None, Vg=None):
    """Gradients (dQ, dK, dV), float64 [B, H, n, d], of ``oracle_longformer``
    (``terms``: as for ``oracle_bigbird_bwd``).

    With the separate projections for global attention (``Qg``, ``Kg``,
    ``Vg``), the global rows depend only on the g set and the other rows only
    on Q, K, V, so the gradients split by rows: returns (dQ, dK, dV, dQg, dKg,
    dVg), each set summed over its own rows; with ``terms``, ((six gradients),
    six (sum |term|, sqrt(sum term^2)) pairs).
    """
    if Qg is not None:
        return _longformer_bwd_split(Q, K, V, dO, window, global_idx, key_mask, dilation, causal,
                                     row_chunk, Qg, Kg, Vg, terms)
    Q, K, V, dO = _as_f64(Q), _as_f64(K), _as_f64(V), _as_f64(dO)
    B, H, n, d = Q.shape
    dil = np.zeros(H, dtype=np.int64) if dilation is None else np.asarray(dilation, dtype=np.int64)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    T = [[np.zeros_like(Q), np.zeros_like(Q)] for _ in range(3)] if terms else None
    for h in range(H):
        for beta in range(B):
            kv = None if key_mask is None else np.asarray(key_mask[beta]) != 0

            def mask_of_rows(rr):
                return _apply_validity(longformer_allowed(n, window, global_idx, rr, dilation=dil[h],
                                                          causal=causal), rr, kv)

            res = _grads_over_rows(Q[beta, h], K[beta, h], V[beta, h], dO[beta, h], mask_of_rows, n,
                                   row_chunk, terms)
            if terms:
                res, tt = res
                for which in range(3):
                    for kind in range(2):
                        T[which][kind][beta, h] = tt[which][kind]
            dQ[beta, h], dK[beta, h], dV[beta, h] = res
    return ((dQ, dK, dV), T) if terms else (dQ, dK, dV)


def _longformer_bwd_split(Q, K, V, dO, window, global_idx, key_mask, dilation, causal, row_chunk, Qg, Kg, Vg,
                          terms=False):
    """Separate projections: rows of global tokens against (Qg, Kg, Vg), the
    other rows against (Q, K, V); each row set's mask is the row's usual mask."""
    Q, K, V, dO = _as_f64(Q), _as_f64(K), _as_f64(V), _as_f64(dO)
    Qg, Kg, Vg = _as_f64(Qg), _as_f64(Kg), _as_f64(Vg)
    B, H, n, d = Q.shape
    dil = np.zeros(H, dtype=np.int64) if dilation is None else np.asarray(dilation, dtype=np.int64)
    is_global = np.zeros(n, dtype=bool)
    is_global[np.asarray(global_idx, dtype=np.int64)] = True
    out = [np.zeros_like(Q) for _ in range(6)]
    ta = [np.zeros_like(Q) for _ in range(6)]  # sum |term|
    t2 = [np.zeros_like(Q) for _ in range(6)]  # sum term^2
    for h in range(H):
        for beta in range(B):
            kv = None if key_mask is None else np.asarray(key_mask[beta]) != 0
            for sel, (q, k, v), base in ((~is_global, (Q, K, V), 0), (is_global, (Qg, Kg, Vg), 3)):
                rows = np.nonzero(sel)[0]
                for c0 in range(0, len(rows), row_chunk):
                    rr = rows[c0:c0 + row_chunk]
                    mask = _apply_validity(longformer_allowed(n, window, global_idx, rr, dilation=dil[h],
                                                              causal=causal), rr, kv)
                    args = (q[beta, h, rr], k[beta, h], v[beta, h], mask, dO[beta, h, rr])
                    dq, dk, dv = masked_attention_grads(*args)
                    out[base][beta, h, rr] = dq
                    out[base + 1][beta, h] += dk
                    out[base + 2][beta, h] += dv
                    if terms:
                        (qa, qr), (ka, kr), (va, vr) = masked_attention_grad_terms(*args)
                        ta[base][beta, h, rr], t2[base][beta, h, rr] = qa, qr * qr
                        ta[base + 1][beta, h] += ka
                        t2[base + 1][beta, h] += kr * kr
                        ta[base + 2][beta, h] += va
                        t2[base + 2][beta, h] += vr * vr
    if not terms:
        return tuple(out)
    return tuple(out), tuple((ta[i], np.sqrt(t2[i])) for i in range(6))


# ---------------------------------------------------------------------------
# Work accounting: attended (valid query, allowed valid key) pairs
# ---------------------------------------------------------------------------

def bigbird_attended_pairs(n, b, g, w, rand_table, key_mask=None, B=1):
    """Number of True entries of M summed over batch entries and heads."""
    rand_table = np.asarray(rand_table)
    H = rand_table.shape[0]
    total = 0
    for h in range(H):
        blk = bigbird_block_allowed(n // b, g, w, rand_table[h])
        for beta in range(B):
            if key_mask is None:
                total += int(blk.sum()) * b * b
            else:
                kv = np.asarray(key_mask[beta]) != 0
                per_blk = kv.reshape(n // b, b).sum(axis=1).astype(np.int64)
                total += int(per_blk @ blk.astype(np.int64) @ per_blk)
    return total


def longformer_attended_pairs(n, window, global_idx, key_mask=None, B=1, H=1, dilation=None,
                              causal=False):
    dil = np.zeros(H, dtype=np.int64) if dilation is None else np.asarray(dilation, dtype=np.int64)
    total = 0
    for h in range(H):
        for beta in range(B):
            kv = None if key_mask is None else np.asarray(key_mask[beta]) != 0
            for c0 in range(0, n, 1024):
                rr = np.arange(c0, min(n, c0 + 1024))
                total += int(_apply_validity(
                    longformer_allowed(n, window, global_idx, rr, dilation=dil[h], causal=causal), rr, kv).sum())
    return total
