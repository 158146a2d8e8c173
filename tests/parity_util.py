"""Shared helpers for the GPU parity tests: run a case through the C ABI and
compare with the float64 oracle on the same seeded inputs."""

import numpy as np
import torch

import block_sparse_long_bigbird_gb300 as sa
from block_sparse_long_bigbird_gb300.inputs import make_qkv
from oracle import bigbird_random_table, oracle_bigbird, oracle_longformer

PATHS = ["simt", "tc"]


def pattern_table(seed, H, n, b, g, w, r):
    """The random-block table the oracle side draws itself, as an int32 tensor.

    Every GPU case feeds this table to both sides, so the oracle never takes
    an input made by the product. The product's host pattern builder
    (``build_bigbird_pattern``) must produce the same table bit for bit, which
    re-checks the builder at every shape a GPU test uses: "Big Bird", App. D
    (Fig. 6 caption) has the blockified product give exactly the sparse
    pattern, so the pattern is compared against an independent statement of
    it, not only through its effect on the output.
    """
    ref = bigbird_random_table(seed, H, n, b, g, w, r)
    got = sa.build_bigbird_pattern(seed, H, n, b, g, w, r).numpy()
    assert got.dtype == ref.dtype and np.array_equal(got, ref), \
        f"build_bigbird_pattern differs from the oracle's table at {(seed, H, n, b, g, w, r)}"
    return torch.from_numpy(ref.copy())


def set_path(path):
    sa.set_option(sa.SA_OPT_FORCE_SIMT, 1 if path == "simt" else 0)


def gpu_bigbird(Q, K, V, b, g, w, r, table, key_mask=None, path="tc"):
    dev = torch.device("cuda:0")
    set_path(path)
    try:
        O = sa.bigbird_attn_fwd(Q.to(dev), K.to(dev), V.to(dev), b, g, w, r,
                                table.to(dev) if r > 0 else None,
                                None if key_mask is None else key_mask.to(dev))
        torch.cuda.synchronize()
        assert sa.get_last_device_status() == 0
    finally:
        set_path("tc")
    return O


def gpu_longformer(Q, K, V, window, gidx, key_mask=None, path="tc", dilation=None, causal=False):
    dev = torch.device("cuda:0")
    set_path(path)
    try:
        O = sa.longformer_attn_fwd(Q.to(dev), K.to(dev), V.to(dev), window,
                                   None if gidx is None else gidx.to(dev),
                                   None if key_mask is None else key_mask.to(dev),
                                   dilation=None if dilation is None else
                                   torch.as_tensor(dilation, dtype=torch.int32).to(dev),
                                   causal=causal)
        torch.cuda.synchronize()
        assert sa.get_last_device_status() == 0
    finally:
        set_path("tc")
    return O


def assert_close(got, ref, tol_max, tol_mean, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= tol_max and err.mean() <= tol_mean, \
        f"{what}: max|err| {err.max():.3e} (tol {tol_max}), mean|err| {err.mean():.3e} (tol {tol_mean})"
    return err.max(), err.mean()


def bigbird_case(B, H, n, d, b, g, w, r, dtype="bf16", sigma=1.0, cfg_id=50, key_mask=None,
                 seed=0, path="tc", rows=None, heads=None, tol=(2e-2, 2e-3)):
    """Run BigBird on the GPU and compare (all rows, or `rows` of the `heads` (beta, h) pairs)."""
    Q, K, V = make_qkv(B, H, n, d, dtype, sigma=sigma, cfg_id=cfg_id)
    table = pattern_table(seed, H, n, b, g, w, r)
    O = gpu_bigbird(Q, K, V, b, g, w, r, table, key_mask, path).float().cpu()
    heads = heads if heads is not None else [(beta, h) for beta in range(B) for h in range(H)]
    for beta, h in heads:
        km = None if key_mask is None else key_mask[beta:beta + 1].numpy()
        ref = oracle_bigbird(Q[beta:beta + 1, h:h + 1], K[beta:beta + 1, h:h + 1], V[beta:beta + 1, h:h + 1],
                             b, g, w, table.numpy()[h:h + 1], key_mask=km, rows=rows)[0, 0]
        got = O[beta, h].numpy() if rows is None else O[beta, h].numpy()[np.asarray(rows)]
        assert_close(got, ref, *tol, what=f"bigbird beta={beta} h={h}")
        if key_mask is not None:
            pad = np.nonzero(key_mask[beta].numpy() == 0)[0]
            if rows is not None:
                pad = np.intersect1d(pad, np.asarray(rows))
            assert np.all(O[beta, h].numpy()[pad] == 0.0), "padded query rows must be exactly 0"
    return O


def longformer_case(B, H, n, d, window, gidx, dtype="bf16", cfg_id=60, key_mask=None, path="tc",
                    rows=None, heads=None, tol=(2e-2, 2e-3), sigma=1.0, dilation=None, causal=False):
    Q, K, V = make_qkv(B, H, n, d, dtype, sigma=sigma, cfg_id=cfg_id)
    O = gpu_longformer(Q, K, V, window, gidx, key_mask, path, dilation, causal).float().cpu()
    heads = heads if heads is not None else [(beta, h) for beta in range(B) for h in range(H)]
    g_np = np.zeros(0, dtype=np.int64) if gidx is None else gidx.numpy()
    for beta, h in heads:
        km = None if key_mask is None else key_mask[beta:beta + 1].numpy()
        ref = oracle_longformer(Q[beta:beta + 1, h:h + 1], K[beta:beta + 1, h:h + 1], V[beta:beta + 1, h:h + 1],
                                window, g_np, key_mask=km, rows=rows,
                                dilation=None if dilation is None else [dilation[h]], causal=causal)[0, 0]
        got = O[beta, h].numpy() if rows is None else O[beta, h].numpy()[np.asarray(rows)]
        assert_close(got, ref, *tol, what=f"longformer beta={beta} h={h}")
        if key_mask is not None:
            pad = np.nonzero(key_mask[beta].numpy() == 0)[0]
            if rows is not None:
                pad = np.intersect1d(pad, np.asarray(rows))
            assert np.all(O[beta, h].numpy()[pad] == 0.0), "padded query rows must be exactly 0"
    return O


def sampled_bigbird_rows(n, b, g, n_random_blocks=8, seed=0):
    """Global rows, first/second-to-last/last query blocks and seeded random blocks."""
    nb = n // b
    rng = np.random.default_rng(seed)
    blocks = set(range(min(g, nb))) | {min(g, nb - 1), nb - 2, nb - 1}
    blocks |= set(int(x) for x in rng.choice(np.arange(nb), size=min(n_random_blocks, nb), replace=False))
    return np.concatenate([np.arange(j * b, (j + 1) * b) for j in sorted(blocks) if 0 <= j < nb])


# --------------------------------------------------------------------------- backward
# Gradient tolerance, derived from the arithmetic (the backward has no stated
# bound). The bf16 tensor-core path rounds each factor P_ij (for dV) and dS_ij
# (for dQ, dK) to bf16 before the products, a relative error of at most 2^-9
# per term, and rounds the output (at most 2^-8 relative; 2^-9 on average).
# With A = sum |term| and R = sqrt(sum term^2) of the element's sum (from the
# oracle), every element obeys |err| <= 2^-8 A + 2^-8 |ref| (twice the
# worst case of the factor rounding, for the fp32 arithmetic around it), and
# independent roundings keep the mean near 2^-9 R / sqrt(3) + 2^-10 |ref|:
# the mean of |err| must stay below the mean of 2^-9 (R + |ref|). fp32 inputs
# run exact fp32 arithmetic: the forward's 1e-4 applied in units of the
# reference gradient's RMS, plus 1e-5 relative, and the mean error within a
# tenth of the max bound's RMS part (the forward's max / mean ratio).
FP32_GRAD_TOL = (1e-4, 1e-5)
FP32_GRAD_MEAN_TOL = 1e-5


def assert_close_grad(got, ref, dtype, terms=None, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite gradient"
    err = np.abs(got - ref)
    rms = max(float(np.sqrt(np.mean(ref ** 2))), 1e-30)
    if dtype == "bf16":
        A, R = (np.asarray(t, dtype=np.float64) for t in terms)
        bound = 2.0 ** -8 * (A + np.abs(ref)) + 1e-6 * rms
        mean_bound = float(np.mean(2.0 ** -9 * (R + np.abs(ref))))
        ratio = err / bound
        assert ratio.max() <= 1.0 and err.mean() <= mean_bound, \
            f"{what}: max err/bound {ratio.max():.3f}, mean|err| {err.mean():.3e} (bound {mean_bound:.3e}), " \
            f"max|err|/rms {err.max() / rms:.3e}"
        return ratio.max(), (err.mean() / mean_bound) if mean_bound > 0 else 0.0
    tmax, trel = FP32_GRAD_TOL
    excess = err - (tmax * rms + trel * np.abs(ref))
    assert excess.max() <= 0, f"{what}: max|err|/rms {err.max() / rms:.3e} (tol {tmax} rms + {trel} |ref|)"
    assert err.mean() <= FP32_GRAD_MEAN_TOL * rms, \
        f"{what}: mean|err|/rms {err.mean() / rms:.3e} (tol {FP32_GRAD_MEAN_TOL})"
    return err.max() / rms, err.mean() / rms


def gpu_bigbird_bwd(Q, K, V, dO, b, g, w, r, table, key_mask=None, path="tc"):
    """Forward then backward through the library; returns (O, dQ, dK, dV) on the CPU."""
    dev = torch.device("cuda:0")
    set_path(path)
    try:
        q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
        tab = table.to(dev) if r > 0 else None
        km = None if key_mask is None else key_mask.to(dev)
        O = sa.bigbird_attn_fwd(q, k, v, b, g, w, r, tab, km)
        dQ, dK, dV = sa.bigbird_attn_bwd(q, k, v, do, b, g, w, r, tab, km)
        torch.cuda.synchronize()
        assert sa.get_last_device_status() == 0
    finally:
        set_path("tc")
    return tuple(t.float().cpu() for t in (O, dQ, dK, dV))


def gpu_longformer_bwd(Q, K, V, dO, window, gidx, key_mask=None, path="tc", dilation=None, causal=False):
    dev = torch.device("cuda:0")
    set_path(path)
    try:
        q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
        gi = None if gidx is None else gidx.to(dev)
        km = None if key_mask is None else key_mask.to(dev)
        dil = None if dilation is None else torch.as_tensor(dilation, dtype=torch.int32).to(dev)
        O = sa.longformer_attn_fwd(q, k, v, window, gi, km, dilation=dil, causal=causal)
        dQ, dK, dV = sa.longformer_attn_bwd(q, k, v, do, window, gi, km, dilation=dil, causal=causal)
        torch.cuda.synchronize()
        assert sa.get_last_device_status() == 0
    finally:
        set_path("tc")
    return tuple(t.float().cpu() for t in (O, dQ, dK, dV))


def _check_grads(got, ref, terms, dtype, key_mask, beta, what):
    for name, gg, rr, tt in zip(("dQ", "dK", "dV"), got, ref, terms):
        assert_close_grad(gg, rr, dtype, terms=tt, what=f"{what} {name}")
    if key_mask is not None:
        pad = np.nonzero(key_mask[beta].numpy() == 0)[0]
        for name, gg in zip(("dQ", "dK", "dV"), got):
            assert np.all(gg[pad] == 0.0), f"{what}: padded positions must have {name} exactly 0"


def bigbird_bwd_case(B, H, n, d, b, g, w, r, dtype="bf16", sigma=1.0, cfg_id=70, key_mask=None, seed=0,
                     path="tc", heads=None):
    from block_sparse_long_bigbird_gb300.inputs import make_grad_out
    from oracle import oracle_bigbird_bwd

    Q, K, V = make_qkv(B, H, n, d, dtype, sigma=sigma, cfg_id=cfg_id)
    dO = make_grad_out(B, H, n, d, dtype, cfg_id=cfg_id)
    table = pattern_table(seed, H, n, b, g, w, r)
    _, dQ, dK, dV = gpu_bigbird_bwd(Q, K, V, dO, b, g, w, r, table, key_mask, path)
    heads = heads if heads is not None else [(beta, h) for beta in range(B) for h in range(H)]
    for beta, h in heads:
        sl = (slice(beta, beta + 1), slice(h, h + 1))
        km = None if key_mask is None else key_mask[beta:beta + 1].numpy()
        ref, terms = oracle_bigbird_bwd(Q[sl], K[sl], V[sl], dO[sl], b, g, w, table.numpy()[h:h + 1],
                                        key_mask=km, terms=True)
        _check_grads([t[beta, h].numpy() for t in (dQ, dK, dV)], [t[0, 0] for t in ref],
                     [(a[0, 0], r[0, 0]) for a, r in terms], dtype, key_mask, beta, f"bigbird bwd beta={beta} h={h}")
    return dQ, dK, dV


def longformer_bwd_case(B, H, n, d, window, gidx, dtype="bf16", cfg_id=80, key_mask=None, path="tc",
                        heads=None, sigma=1.0, dilation=None, causal=False):
    from block_sparse_long_bigbird_gb300.inputs import make_grad_out
    from oracle import oracle_longformer_bwd

    Q, K, V = make_qkv(B, H, n, d, dtype, sigma=sigma, cfg_id=cfg_id)
    dO = make_grad_out(B, H, n, d, dtype, cfg_id=cfg_id)
    _, dQ, dK, dV = gpu_longformer_bwd(Q, K, V, dO, window, gidx, key_mask, path, dilation, causal)
    heads = heads if heads is not None else [(beta, h) for beta in range(B) for h in range(H)]
    g_np = np.zeros(0, dtype=np.int64) if gidx is None else gidx.numpy()
    for beta, h in heads:
        sl = (slice(beta, beta + 1), slice(h, h + 1))
        km = None if key_mask is None else key_mask[beta:beta + 1].numpy()
        ref, terms = oracle_longformer_bwd(Q[sl], K[sl], V[sl], dO[sl], window, g_np, key_mask=km,
                                           dilation=None if dilation is None else [dilation[h]], causal=causal,
                                           terms=True)
        _check_grads([t[beta, h].numpy() for t in (dQ, dK, dV)], [t[0, 0] for t in ref],
                     [(a[0, 0], r[0, 0]) for a, r in terms], dtype, key_mask, beta,
                     f"longformer bwd beta={beta} h={h}")
    return dQ, dK, dV
