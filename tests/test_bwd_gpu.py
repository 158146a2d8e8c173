"""GPU parity of the backward pass (dQ, dK, dV) against the float64 oracle.

The bound (``parity_util.assert_close_grad``) is derived from the arithmetic:
for bf16 inputs each element's error stays within 2^-8 of the sum of the
magnitudes of its terms plus its own magnitude, and the mean error within
2^-9 of the terms' root-sum-square plus magnitude (term sizes from the
oracle); fp32 inputs use 1e-4 of the reference gradient's RMS plus 1e-5
relative (``FP32_GRAD_TOL``) per element and 1e-5 of the RMS on the mean
(``FP32_GRAD_MEAN_TOL``). Every case runs through the C ABI (the forward,
then the backward at the same inputs).
"""

import numpy as np
import pytest
import torch

import block_sparse_long_bigbird_gb300 as sa
from block_sparse_long_bigbird_gb300.inputs import make_grad_out, make_key_mask, make_qkv, make_random_key_mask
from parity_util import PATHS, bigbird_bwd_case, gpu_bigbird_bwd, longformer_bwd_case, pattern_table

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    sa._lib.lib()
    yield
    sa.set_option(sa.SA_OPT_FORCE_SIMT, 0)


BIGBIRD_BWD = [
    # B, H, n,    d,   b,   g, w, r
    (2, 2, 1024, 64, 64, 2, 3, 3),
    (1, 2, 192, 64, 64, 1, 3, 3),      # nb = 3
    (1, 2, 1024, 128, 128, 2, 3, 3),
    (1, 1, 768, 128, 64, 1, 5, 2),
    (1, 2, 1024, 64, 128, 2, 3, 3),
    (2, 1, 640, 64, 64, 0, 1, 0),      # block-diagonal
    (1, 1, 512, 64, 64, 1, 1, 8),      # r >= nb: full attention
]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case", BIGBIRD_BWD, ids=lambda c: "B{}H{}n{}d{}b{}g{}w{}r{}".format(*c))
def test_bigbird_bwd_small(case, path):
    bigbird_bwd_case(*case, dtype="bf16", path=path)


@pytest.mark.parametrize("d,b", [(64, 64), (128, 128)])
def test_bigbird_bwd_fp32(d, b):
    bigbird_bwd_case(1, 2, 1024, d, b, 2, 3, 3, dtype="fp32", path="simt")


@pytest.mark.parametrize("path", PATHS)
def test_bigbird_bwd_prefix_padding(path):
    B, n = 2, 2048
    bigbird_bwd_case(B, 2, n, 64, 64, 2, 3, 3, key_mask=make_key_mask(B, n), path=path)


@pytest.mark.parametrize("path", PATHS)
def test_bigbird_bwd_random_padding_d128(path):
    B, n = 1, 1024
    bigbird_bwd_case(B, 2, n, 128, 128, 2, 3, 3, key_mask=make_random_key_mask(B, n), path=path)


@pytest.mark.parametrize("path", PATHS)
def test_bigbird_bwd_headline_sampled_heads(path):
    """B=8 H=12 n=4096 d=64 (the headline forward workload), two heads compared in full."""
    bigbird_bwd_case(8, 12, 4096, 64, 64, 2, 3, 3, path=path, heads=[(0, 0), (7, 11)], cfg_id=71)


LONGFORMER_BWD = [
    # B, H, n,    d,   window, globals,        dilation, causal
    (2, 2, 1000, 64, 128, [0, 5, 500], None, False),
    (1, 2, 777, 128, 64, [3, 400, 776], None, False),
    (1, 2, 1000, 64, 96, [0, 5, 500], [0, 2], False),
    (1, 2, 1000, 64, 128, [0, 5, 500], None, True),
    (1, 2, 900, 64, 64, [1, 450], [1, 3], True),
    (1, 1, 300, 64, 0, [], None, False),           # window 0, no globals: each token sees itself
    (1, 1, 256, 64, 1024, [], None, False),        # window wider than the sequence: full attention
]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case", LONGFORMER_BWD, ids=lambda c: "B{}H{}n{}d{}win{}dil{}c{}".format(
    *c[:5], c[6], int(c[7])))
def test_longformer_bwd_small(case, path):
    B, H, n, d, window, globals_, dilation, causal = case
    gidx = torch.tensor(globals_, dtype=torch.int32) if globals_ else None
    longformer_bwd_case(B, H, n, d, window, gidx, path=path, dilation=dilation, causal=causal)


def test_longformer_bwd_fp32_padded():
    B, n = 2, 1000
    longformer_bwd_case(B, 2, n, 64, 128, torch.tensor([0, 7, 640], dtype=torch.int32), dtype="fp32",
                        key_mask=make_key_mask(B, n), path="simt", dilation=[0, 1], causal=False)


@pytest.mark.parametrize("path", PATHS)
def test_longformer_bwd_headline_sampled_heads(path):
    """B=4 H=12 n=4096 d=64 window 512, globals {0..15}; two heads compared in full."""
    longformer_bwd_case(4, 12, 4096, 64, 512, torch.arange(16, dtype=torch.int32), path=path,
                        heads=[(0, 0), (3, 11)], cfg_id=81)


@pytest.mark.parametrize("path", PATHS)
def test_bwd_is_deterministic(path):
    B, H, n, d = 2, 2, 1024, 64
    Q, K, V = make_qkv(B, H, n, d, "bf16", cfg_id=72)
    dO = make_grad_out(B, H, n, d, "bf16", cfg_id=72)
    table = pattern_table(0, H, n, 64, 2, 3, 3)
    first = gpu_bigbird_bwd(Q, K, V, dO, 64, 2, 3, 3, table, path=path)
    second = gpu_bigbird_bwd(Q, K, V, dO, 64, 2, 3, 3, table, path=path)
    for a, b in zip(first, second):
        assert torch.equal(a, b)


def test_bwd_bad_random_entry_latches_status():
    dev = torch.device("cuda:0")
    B, H, n, d = 1, 1, 512, 64
    Q, K, V = (t.to(dev) for t in make_qkv(B, H, n, d, "bf16", cfg_id=73))
    dO = make_grad_out(B, H, n, d, "bf16", cfg_id=73).to(dev)
    table = pattern_table(0, H, n, 64, 2, 3, 3)
    O = sa.bigbird_attn_fwd(Q, K, V, 64, 2, 3, 3, table.to(dev))
    torch.cuda.synchronize()
    assert sa.get_last_device_status() == 0
    table[0, 4, 0] = 99  # out of range: skipped and latched
    sa.bigbird_attn_bwd(Q, K, V, dO, 64, 2, 3, 3, table.to(dev))
    assert sa.get_last_device_status() == sa._lib.SA_ERR_BAD_INDEX
    assert sa.get_last_device_status() == 0


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("causal,dilation", [(False, None), (True, [0, 2])])
def test_longformer_gproj_bwd(path, causal, dilation):
    """Six gradients of the separate-projection forward: non-global rows into
    Q, K, V, global rows into Qg, Kg, Vg."""
    from oracle import oracle_longformer_bwd
    from parity_util import assert_close_grad, set_path
    dev = torch.device("cuda:0")
    B, H, n, d, window = 2, 2, 1000, 64, 128
    gidx = torch.tensor([0, 5, 500, 999], dtype=torch.int32)
    km = make_key_mask(B, n)
    Q, K, V = make_qkv(B, H, n, d, "bf16", cfg_id=110)
    Qg, Kg, Vg = make_qkv(B, H, n, d, "bf16", cfg_id=111)
    dO = make_grad_out(B, H, n, d, "bf16", cfg_id=110)
    set_path(path)
    try:
        dil = None if dilation is None else torch.tensor(dilation, dtype=torch.int32, device=dev)
        grads = sa.longformer_attn_bwd_gproj(*(t.to(dev) for t in (Q, K, V, Qg, Kg, Vg, dO)), window,
                                             gidx.to(dev), km.to(dev), dilation=dil, causal=causal)
        torch.cuda.synchronize()
        assert sa.get_last_device_status() == 0
    finally:
        set_path("tc")
    grads = [t.float().cpu().numpy() for t in grads]
    for beta in range(B):
        for h in range(H):
            sl = (slice(beta, beta + 1), slice(h, h + 1))
            refs, terms = oracle_longformer_bwd(Q[sl], K[sl], V[sl], dO[sl], window, gidx.numpy(),
                                                key_mask=km[beta:beta + 1].numpy(),
                                                dilation=None if dilation is None else [dilation[h]], causal=causal,
                                                Qg=Qg[sl], Kg=Kg[sl], Vg=Vg[sl], terms=True)
            for i, name in enumerate(("dQ", "dK", "dV", "dQg", "dKg", "dVg")):
                assert_close_grad(grads[i][beta, h], refs[i][0, 0], "bf16",
                                  terms=(terms[i][0][0, 0], terms[i][1][0, 0]), what=f"gproj {name} b={beta} h={h}")


def _sampled_bwd_check(wl_name, path, heads, kblocks, seed):
    """Full-size backward in the bench's configuration: dQ on sampled query
    blocks, dK and dV on sampled non-global key blocks, against the exact
    sampled oracle, within the bf16 rounding bound."""
    from block_sparse_long_bigbird_gb300.workloads import WORKLOADS
    from oracle import oracle_bigbird_bwd_sampled
    from parity_util import assert_close_grad, sampled_bigbird_rows, set_path
    wl = WORKLOADS[wl_name]
    dev = torch.device("cuda:0")
    Q, K, V = make_qkv(wl.B, wl.H, wl.n, wl.d, "bf16", sigma=wl.sigma, cfg_id=wl.cfg_id)
    dO = make_grad_out(wl.B, wl.H, wl.n, wl.d, "bf16", cfg_id=wl.cfg_id)
    table = pattern_table(wl.seed, wl.H, wl.n, wl.b, wl.g, wl.w, wl.r)
    km = make_key_mask(wl.B, wl.n) if wl.padded else None
    set_path(path)
    try:
        grads = sa.bigbird_attn_bwd(*(t.to(dev) for t in (Q, K, V, dO)), wl.b, wl.g, wl.w, wl.r, table.to(dev),
                                    None if km is None else km.to(dev))
        torch.cuda.synchronize()
        assert sa.get_last_device_status() == 0
    finally:
        set_path("tc")
    grads = [t.float().cpu().numpy() for t in grads]
    rows = sampled_bigbird_rows(wl.n, wl.b, wl.g, n_random_blocks=3, seed=seed)
    keys = np.concatenate([np.arange(k * wl.b, (k + 1) * wl.b) for k in kblocks])
    for beta, h in heads:
        (dq, tq), (dk, tk), (dv, tv) = oracle_bigbird_bwd_sampled(
            Q[beta, h], K[beta, h], V[beta, h], dO[beta, h], wl.b, wl.g, wl.w, table.numpy()[h], rows, kblocks,
            key_valid=None if km is None else km[beta].numpy())
        assert_close_grad(grads[0][beta, h][rows], dq, "bf16", terms=tq, what=f"{wl_name} dQ {beta},{h}")
        assert_close_grad(grads[1][beta, h][keys], dk, "bf16", terms=tk, what=f"{wl_name} dK {beta},{h}")
        assert_close_grad(grads[2][beta, h][keys], dv, "bf16", terms=tv, what=f"{wl_name} dV {beta},{h}")


def test_bigbird_bwd_n65536_d128_sampled():
    _sampled_bwd_check("bigbird_bwd_bf16_n65536_d128", "tc", [(0, 0), (0, 13)], [5, 200, 511], seed=7)


@pytest.mark.parametrize("path", PATHS)
def test_bigbird_bwd_n16384_padded_sampled(path):
    from block_sparse_long_bigbird_gb300.workloads import WORKLOADS, Workload
    import dataclasses
    base = WORKLOADS["bigbird_bf16_n16384_padded"]
    WORKLOADS.setdefault("_bwd_n16384_padded", dataclasses.replace(base, name="_bwd_n16384_padded", grad=True))
    _sampled_bwd_check("_bwd_n16384_padded", path, [(0, 0), (1, 15)], [3, 100, 255], seed=8)
