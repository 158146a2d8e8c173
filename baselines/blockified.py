"""The pages' own dense-operation formulation of sparse attention, in plain
PyTorch: a comparison baseline that runs on the same GPU as the library and is
timed beside it. It is not part of the library and imports nothing from it.

BigBird ("Big Bird", App. D, Eq. (13), Fig. 4-6; the BigBird blog summary,
Sec. 4.2 "implementation tricks"): the queries are reshaped into blocks
[nb, b, d]; each query block gets its own key tensor K'' of (g + w + r) blocks,
the concatenation of
  * the g global key blocks (the same for every query block),
  * w copies of the blocked keys, each rolled by one offset of the sliding
    window (copy o holds block j + o at position j), and
  * the r random key blocks of that query block, gathered;
one batched dense product then scores every query block against its K'' at
once, and the same layout of V gives the output. The global query blocks
(rows of blocks 0..g-1, which see every key) are computed by a direct dense
product against all keys.

Longformer ("Longformer", App. A, the "chunks" implementation; Sec. 3.1 for
the pattern): Q and K are cut into chunks of w = window tokens that overlap by
w / 2; one batched product per chunk gives a w x w score block, of which only
the band diagonals are kept. Every query row lies in two chunks, and its
2 * (w / 2) + 1 band keys are split between them, so a row's softmax runs over
its part of both chunks plus the global keys. Tokens with global attention
attend all keys through a direct dense product. Like the pages' chunks
version, this handles the plain (non-dilated) window; autoregressive mode is
a further mask on the same blocks.

Where the pages leave a step open the library's reading is used, so that the
two compute the same function:
  * the window is clipped at the sequence ends: a rolled copy that wraps
    around (block j + o outside [0, nb)) is masked, not attended;
  * a key block that appears in two parts of K'' (a window block that is also
    global, or a random entry that repeats a global or window block or an
    earlier random entry) is attended once: the later copy is masked;
  * key padding removes keys, and a padded query row outputs zeros; a row with
    no allowed key outputs zeros.

Precision: the products run in the input dtype on the tensor cores (cuBLAS),
so the scores are rounded to it; the softmax runs in float32 (float64 for
float64 inputs), and P is cast back to the input dtype for the P V product, as
a model written with these dense operations would do.
"""

import math

import torch


def _masked_softmax(scores, allowed, scale, out_dtype, may_be_empty):
    """Row softmax of scale * `scores` over `allowed`, computed in float32
    (float64 for float64 inputs) and returned in `out_dtype`. With
    `may_be_empty`, rows with nothing allowed give zeros."""
    acc = torch.promote_types(scores.dtype, torch.float32)
    s = scores.mul_(scale).masked_fill_(~allowed, float("-inf"))
    p = torch.softmax(s, dim=-1, dtype=acc)
    if may_be_empty:
        p = p.nan_to_num_(0.0)
    return p.to(out_dtype)


def bigbird_blockified(Q, K, V, b, g, w, r, rand_table, key_mask=None):
    """BigBird-ITC attention [B, H, n, d] by the blockified dense operations.

    Q, K, V: [B, H, n, d] on one device, n a multiple of b. rand_table: int
    [H, n // b, r] (-1: no block) or None when r = 0. key_mask: [B, n] (nonzero
    = valid token) or None.
    """
    B, H, n, d = Q.shape
    if n % b != 0:
        raise ValueError("n must be a multiple of the block size b")
    nb = n // b
    half = w // 2
    dev = Q.device
    scale = 1.0 / math.sqrt(d)
    Qb = Q.reshape(B, H, nb, b, d)
    Kb = K.reshape(B, H, nb, b, d)
    Vb = V.reshape(B, H, nb, b, d)
    j = torch.arange(nb, device=dev)

    # --- K'' and V'': [B, H, nb, g + w + r, b, d]
    offs = list(range(-half, half + 1))
    parts_k = [Kb[:, :, :g].unsqueeze(2).expand(B, H, nb, g, b, d)]
    parts_v = [Vb[:, :, :g].unsqueeze(2).expand(B, H, nb, g, b, d)]
    parts_k.append(torch.stack([torch.roll(Kb, shifts=-o, dims=2) for o in offs], dim=3))
    parts_v.append(torch.stack([torch.roll(Vb, shifts=-o, dims=2) for o in offs], dim=3))
    # key block of every column block, and whether that column block is attended
    win = j[:, None] + j.new_tensor(offs)[None, :]
    cols = [j.new_tensor(range(g)).expand(nb, g), win % nb]  # the roll wraps around
    ok = [torch.ones(nb, g, dtype=torch.bool, device=dev), (win >= 0) & (win < nb) & (win >= g)]
    cols = [c.unsqueeze(0).expand(H, -1, -1) for c in cols]
    ok = [c.unsqueeze(0).expand(H, -1, -1) for c in ok]
    if r > 0 and rand_table is not None:
        rt = rand_table.to(device=dev, dtype=torch.long)
        hh = torch.arange(H, device=dev)[:, None, None]
        ri = rt.clamp(min=0)
        parts_k.append(Kb[:, hh, ri])
        parts_v.append(Vb[:, hh, ri])
        rok = (rt >= g) & ((rt - j[None, :, None]).abs() > half)
        # a repeated random entry is attended once
        for t in range(1, rt.shape[-1]):
            rok[..., t] &= (rt[..., t:t + 1] != rt[..., :t]).all(dim=-1)
        cols.append(ri)
        ok.append(rok)
    Kpp = torch.cat(parts_k, dim=3)
    Vpp = torch.cat(parts_v, dim=3)
    ncol = Kpp.shape[3]
    cols = torch.cat(cols, dim=-1)  # [H, nb, ncol]
    ok = torch.cat(ok, dim=-1)
    Kpp = Kpp.reshape(B, H, nb, ncol * b, d)
    Vpp = Vpp.reshape(B, H, nb, ncol * b, d)

    # --- Eq. (13): one batched product for every query block
    A = torch.matmul(Qb, Kpp.transpose(-1, -2))  # [B, H, nb, b, ncol * b]
    allowed = ok.repeat_interleave(b, dim=-1).unsqueeze(0).unsqueeze(3)  # [1, H, nb, 1, ncol * b]
    if key_mask is not None:
        kv = (key_mask.to(dev) != 0).reshape(B, nb, b)
        kvc = kv[:, cols]  # [B, H, nb, ncol, b]
        allowed = allowed & kvc.reshape(B, H, nb, 1, ncol * b)
    P = _masked_softmax(A, allowed, scale, Q.dtype, key_mask is not None)
    O = torch.matmul(P, Vpp).reshape(B, H, n, d)

    # --- the global query blocks: direct product against every key
    if g > 0:
        gr = min(g, nb) * b
        Sg = torch.matmul(Q[:, :, :gr], K.transpose(-1, -2))  # [B, H, gr, n]
        ag = torch.ones(1, 1, 1, n, dtype=torch.bool, device=dev)
        if key_mask is not None:
            ag = (key_mask.to(dev) != 0).reshape(B, 1, 1, n)
        O[:, :, :gr] = torch.matmul(_masked_softmax(Sg, ag, scale, Q.dtype, key_mask is not None), V)
    if key_mask is not None:
        O = O * (key_mask.to(dev) != 0).reshape(B, 1, n, 1).to(O.dtype)
    return O


def longformer_chunks(Q, K, V, window, global_idx, key_mask=None, causal=False):
    """Longformer attention [B, H, n, d] by overlapping chunks.

    window: total window (window // 2 tokens each side, even, >= 2).
    global_idx: int positions with global attention (ascending, in [0, n)),
    possibly empty. key_mask: [B, n] or None. causal: keys after the query are
    masked, global keys included.
    """
    B, H, n, d = Q.shape
    hw = window // 2
    if hw < 1:
        raise ValueError("window must be at least 2")
    dev = Q.device
    scale = 1.0 / math.sqrt(d)
    m = (n + hw - 1) // hw  # query blocks of hw rows
    npad = m * hw
    # pad hw tokens in front and enough behind: chunk c covers tokens
    # [(c - 1) hw, (c + 1) hw), c = 0..m
    tail = npad - n + hw

    def chunks(X):
        Xp = torch.nn.functional.pad(X, (0, 0, hw, tail))
        return Xp.unfold(2, 2 * hw, hw).transpose(-1, -2)  # [B, H, m + 1, 2hw, d]

    Qc, Kc, Vc = chunks(Q), chunks(K), chunks(V)
    Sc = torch.matmul(Qc, Kc.transpose(-1, -2))  # [B, H, m + 1, 2hw, 2hw]
    # query block q sits in chunk q as its second half and in chunk q + 1 as its first half
    S2 = Sc[:, :, :m, hw:, :]  # keys [(q - 1) hw, (q + 1) hw)
    S1 = Sc[:, :, 1:, :hw, :]  # keys [q hw, (q + 2) hw)
    a = torch.arange(hw, device=dev)[:, None]
    t = torch.arange(2 * hw, device=dev)[None, :]
    band2 = (t >= a) & (t < hw)  # keys q hw - hw + t, in [i - hw, q hw)
    band1 = t <= hw + a  # keys q hw + t, in [q hw, i + hw]
    q = torch.arange(m, device=dev)[:, None, None]
    key2 = (q - 1) * hw + t[None]  # [m, 1, 2hw]
    key1 = q * hw + t[None]
    qpos = q * hw + a[None]  # [m, hw, 1]
    gl = torch.as_tensor(global_idx, dtype=torch.long, device=dev).reshape(-1)
    is_g = torch.zeros(n + 2 * hw + npad, dtype=torch.bool, device=dev)
    if gl.numel():
        is_g[gl + hw] = True  # shifted by hw so that key -hw.. index from 0
    if key_mask is not None:
        kvalid = torch.zeros(B, n + 2 * hw + npad, dtype=torch.bool, device=dev)
        kvalid[:, hw:hw + n] = key_mask.to(dev) != 0
    else:
        kvalid = torch.zeros(1, n + 2 * hw + npad, dtype=torch.bool, device=dev)
        kvalid[:, hw:hw + n] = True

    def band_allowed(band, key):
        al = band[None] & ~is_g[key + hw]  # a global key in the band is attended through the global columns
        if causal:
            al = al & (key <= qpos)
        return al.unsqueeze(0) & kvalid[:, key + hw]  # [B or 1, m, hw, 2hw]

    al2 = band_allowed(band2, key2)
    al1 = band_allowed(band1, key1)
    parts = [S2, S1]
    allowed = [al2, al1]
    ng = gl.numel()
    Qblk = torch.nn.functional.pad(Q, (0, 0, 0, npad - n)).reshape(B, H, m, hw, d)
    if ng:
        Kg, Vg = K[:, :, gl], V[:, :, gl]  # [B, H, ng, d]
        Sgc = torch.matmul(Qblk, Kg.unsqueeze(2).transpose(-1, -2))  # [B, H, m, hw, ng]
        alg = torch.ones(1, m, hw, ng, dtype=torch.bool, device=dev)
        if causal:
            alg = alg & (gl[None, None, None, :] <= qpos)
        alg = alg & kvalid[:, gl + hw][:, None, None, :]
        parts.append(Sgc)
        allowed.append(alg)
    S = torch.cat(parts, dim=-1)  # [B, H, m, hw, 4hw (+ ng)]
    al = torch.cat([x.expand(B if x.shape[0] == 1 else x.shape[0], m, hw, x.shape[-1]) for x in allowed], dim=-1)
    rowv = qpos < n
    if key_mask is not None:
        qv = torch.zeros(B, npad, dtype=torch.bool, device=dev)
        qv[:, :n] = key_mask.to(dev) != 0
        rowv = rowv.unsqueeze(0) & qv.reshape(B, m, hw, 1)
    al = (al & rowv).unsqueeze(1)  # [B, 1, m, hw, cols]
    # rows past n have nothing allowed; they are cut off below
    P = _masked_softmax(S, al, scale, Q.dtype, True)
    O = torch.matmul(P[..., :2 * hw], Vc[:, :, :m]) + torch.matmul(P[..., 2 * hw:4 * hw], Vc[:, :, 1:])
    if ng:
        O = O + torch.matmul(P[..., 4 * hw:], Vg.unsqueeze(2))
    O = O.reshape(B, H, npad, d)[:, :, :n].contiguous()

    # --- rows with global attention: direct product against every key
    if ng:
        Sgr = torch.matmul(Q[:, :, gl], K.transpose(-1, -2))  # [B, H, ng, n]
        ag = kvalid[:, hw:hw + n].reshape(-1, 1, 1, n)
        if causal:
            ag = ag & (torch.arange(n, device=dev)[None, :] <= gl[:, None]).reshape(1, 1, ng, n)
        Og = torch.matmul(_masked_softmax(Sgr, ag, scale, Q.dtype, key_mask is not None), V)
        if key_mask is not None:
            Og = Og * (key_mask.to(dev)[:, gl] != 0).reshape(B, 1, ng, 1).to(Og.dtype)
        O[:, :, gl] = Og
    return O
