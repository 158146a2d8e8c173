"""GPU parity: the CUDA kernels (through the C ABI) against the float64 oracle.

Tolerances: bf16 inputs max|err| <= 2e-2 and mean|err| <= 2e-3; fp32 inputs
max|err| <= 1e-4. Every case runs on both kernel families: "tc" (the bf16
tcgen05 pipeline; fp32 always runs on SIMT) and "simt" (the exact SIMT kernels).
"""

import numpy as np
import pytest
import torch

import block_sparse_long_bigbird_gb300 as sa
from block_sparse_long_bigbird_gb300.inputs import make_key_mask, make_qkv, make_random_key_mask
from block_sparse_long_bigbird_gb300.workloads import WORKLOADS
from parity_util import (PATHS, bigbird_case, gpu_bigbird, longformer_case, pattern_table, sampled_bigbird_rows)

pytestmark = pytest.mark.gpu

FP32_TOL = (1e-4, 1e-5)


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    sa._lib.lib()
    yield
    sa.set_option(sa.SA_OPT_FORCE_SIMT, 0)


# ------------------------------------------------------------- BigBird, small full compares

BIGBIRD_SMALL = [
    # B, H, n,    d,   b,   g, w, r
    (2, 3, 512, 64, 64, 2, 3, 3),
    (1, 2, 192, 64, 64, 1, 3, 3),      # nb = 3: odd block count, no random candidates
    (1, 2, 1024, 128, 128, 2, 3, 3),
    (1, 1, 768, 128, 64, 1, 5, 2),
    (1, 2, 1024, 64, 128, 2, 3, 3),
    (2, 1, 640, 64, 64, 0, 1, 0),      # block-diagonal (App. D Eq. 13)
    (1, 1, 512, 64, 64, 1, 1, 8),      # r >= nb: full attention
    (1, 2, 2048, 64, 64, 3, 7, 4),
    (1, 1, 1280, 64, 64, 2, 3, 3),     # nb = 20
]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case", BIGBIRD_SMALL, ids=lambda c: "B{}H{}n{}d{}b{}g{}w{}r{}".format(*c))
def test_bigbird_small(case, path):
    bigbird_case(*case, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_bigbird_fp32_config(path):
    wl = WORKLOADS["bigbird_fp32_n1024"]
    bigbird_case(wl.B, wl.H, wl.n, wl.d, wl.b, wl.g, wl.w, wl.r, dtype="fp32", cfg_id=wl.cfg_id,
                 path=path, tol=FP32_TOL)


@pytest.mark.parametrize("path", PATHS)
def test_bigbird_fp32_d128(path):
    bigbird_case(1, 2, 1024, 128, 128, 2, 3, 3, dtype="fp32", path=path, tol=FP32_TOL)


@pytest.mark.parametrize("path", PATHS)
def test_bigbird_prefix_padding(path):
    B, n = 3, 1024
    km = make_key_mask(B, n, seed=7)
    bigbird_case(B, 2, n, 64, 64, 2, 3, 3, key_mask=km, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_bigbird_random_padding(path):
    B, n = 2, 1024
    km = make_random_key_mask(B, n, seed=8, p_valid=0.7)
    bigbird_case(B, 2, n, 64, 64, 2, 3, 3, key_mask=km, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_bigbird_fully_padded_sequence(path):
    B, n = 2, 512
    km = torch.ones(B, n, dtype=torch.uint8)
    km[1] = 0
    km[0, 300:] = 0
    bigbird_case(B, 1, n, 64, 64, 2, 3, 3, key_mask=km, path=path)


@pytest.mark.parametrize("d,b", [(64, 64), (128, 128)])
@pytest.mark.parametrize("grid", [1, 3])
def test_bigbird_padded_runs_few_ctas(d, b, grid):
    # A persistent CTA meets long runs of fully padded tiles (empty units)
    # right after tiles with work: batch 0 is valid up to token 1000, batch 1
    # is all padding. With one or three CTAs every tile walks those runs.
    B, n = 2, 4096
    km = torch.zeros(B, n, dtype=torch.uint8)
    km[0, :1000] = 1
    sa.set_option(sa.SA_OPT_GRID_CTAS, grid)
    try:
        bigbird_case(B, 2, n, d, b, 2, 3, 3, key_mask=km, path="tc", cfg_id=84)
    finally:
        sa.set_option(sa.SA_OPT_GRID_CTAS, 0)


@pytest.mark.parametrize("grid", [1, 2, 5])
def test_few_ctas_split_sweeps_and_residue_classes(grid):
    # Few persistent CTAs walk every unit kind in sequence: a padded BigBird
    # call whose global tiles are cut into split-KV chunks (2 heads at n = 8192)
    # and a dilated Longformer call on residue-class copies.
    sa.set_option(sa.SA_OPT_GRID_CTAS, grid)
    try:
        km = make_key_mask(1, 8192, seed=41)
        rows = sampled_bigbird_rows(8192, 64, 2, n_random_blocks=4, seed=8)
        bigbird_case(1, 2, 8192, 64, 64, 2, 3, 3, key_mask=km, path="tc", cfg_id=143, rows=rows)
        longformer_case(1, 3, 1200, 64, 96, None, dilation=[0, 1, 3], causal=True, cfg_id=144)
    finally:
        sa.set_option(sa.SA_OPT_GRID_CTAS, 0)


# ------------------------------------------------------------- Longformer, small full compares

LONGFORMER_SMALL = [
    # B, H, n,    d,  window, globals
    (1, 2, 1000, 64, 64, [0, 5, 500, 999]),
    (2, 1, 512, 64, 0, []),
    (1, 1, 256, 64, 1024, [3]),
    (1, 2, 1024, 128, 256, [0, 1, 2, 3]),
    (1, 1, 2048, 64, 512, list(range(16))),
    (1, 1, 777, 64, 100, [776]),
]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case", LONGFORMER_SMALL, ids=lambda c: "B{}H{}n{}d{}win{}".format(*c[:5]))
def test_longformer_small(case, path):
    B, H, n, d, window, G = case
    gidx = torch.tensor(G, dtype=torch.int32) if G else None
    longformer_case(B, H, n, d, window, gidx, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_longformer_many_globals_and_padding(path):
    from block_sparse_long_bigbird_gb300.inputs import make_global_positions

    B, n = 2, 1536
    gidx = make_global_positions(n, 150, seed=5)
    km = make_key_mask(B, n, seed=9)
    longformer_case(B, 1, n, 64, 128, gidx, key_mask=km, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_longformer_fp32(path):
    gidx = torch.tensor([0, 100], dtype=torch.int32)
    longformer_case(1, 1, 640, 64, 64, gidx, dtype="fp32", path=path, tol=FP32_TOL)


@pytest.mark.parametrize("path", PATHS)
def test_longformer_d128_padded(path):
    from block_sparse_long_bigbird_gb300.inputs import make_global_positions

    B, n = 2, 1100
    gidx = make_global_positions(n, 40, seed=11)
    km = make_key_mask(B, n, seed=12)
    longformer_case(B, 1, n, 128, 200, gidx, key_mask=km, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_longformer_every_token_global(path):
    # every row is a global row: the band units store nothing, three global tiles
    n = 300
    gidx = torch.arange(n, dtype=torch.int32)
    longformer_case(1, 2, n, 64, 32, gidx, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_longformer_split_global_rows(path):
    # 12288 keys: the global rows sweep in split-KV chunks (2 heads leave most
    # SMs idle, so the chunks are short); 131 global rows span two global tiles
    from block_sparse_long_bigbird_gb300.inputs import make_global_positions

    n = 12288
    gidx = make_global_positions(n, 131, seed=13)
    rng = np.random.default_rng(14)
    rows = np.unique(np.concatenate([gidx.numpy(), np.arange(0, 200), np.arange(n - 200, n),
                                     rng.choice(n, 300, replace=False)]))
    longformer_case(1, 2, n, 64, 256, gidx, path=path, rows=rows)


# σ = 4 spreads the scaled scores over ~±50: within one 128-key step a row's
# running maximum often rises by more than the lazy-rescale threshold between
# the two 64-key halves, so the rescale of the first half's P runs for some
# rows of a warp and not others. Outputs reach |O| ~ 16 (bf16 half-ulp 1/16
# there), so the tolerance is 8x the σ = 1 one; a first-half P left unscaled
# would be off by a factor of at least 2^8.
WIDE_TOL = (1.6e-1, 1.6e-2)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("d", [64, 128])
def test_bigbird_wide_score_range(path, d):
    bigbird_case(1, 2, 1024, d, 64, 2, 3, 3, sigma=4.0, cfg_id=81, path=path, tol=WIDE_TOL)


@pytest.mark.parametrize("path", PATHS)
def test_bigbird_wide_score_range_padded(path):
    B, n = 2, 1024
    km = make_key_mask(B, n, seed=21, low=200)
    bigbird_case(B, 1, n, 64, 64, 2, 3, 3, sigma=4.0, cfg_id=82, key_mask=km, path=path, tol=WIDE_TOL)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("d", [64, 128])
def test_longformer_wide_score_range(path, d):
    gidx = torch.tensor([0, 5, 500, 999], dtype=torch.int32)
    longformer_case(1, 2, 1000, d, 64, gidx, sigma=4.0, cfg_id=83, path=path, tol=WIDE_TOL)


# ------------------------------------------------- Longformer dilation / autoregressive mode

@pytest.mark.parametrize("path", PATHS)
def test_longformer_dilated_per_head(path):
    gidx = torch.tensor([0, 5, 500], dtype=torch.int32)
    longformer_case(1, 4, 1000, 64, 64, gidx, path=path, dilation=[0, 1, 2, 3], cfg_id=85)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("d", [64, 128])
def test_longformer_causal_padded(path, d):
    B, n = 2, 777
    gidx = torch.tensor([3, 400], dtype=torch.int32)
    km = make_key_mask(B, n, seed=31)
    longformer_case(B, 2, n, d, 100, gidx, key_mask=km, path=path, dilation=[0, 2], causal=True, cfg_id=86)


@pytest.mark.parametrize("path", PATHS)
def test_longformer_causal_no_globals(path):
    longformer_case(1, 2, 1536, 64, 256, None, path=path, causal=True, cfg_id=87)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n,causal", [(3000, False), (3000, True), (3002, False), (6000, True)])
def test_longformer_dilated_residue_classes(d, n, causal):
    # No global tokens, no key mask: dilated heads whose stride divides n run on
    # residue-class copies of Q, K, V (plain windows clipped to each class);
    # n = 3002 leaves strides 3 and 4 on the direct dilated path beside stride 2.
    # Every row of every head is compared.
    longformer_case(1, 4, n, d, 128, None, dilation=[0, 1, 2, 3], causal=causal, cfg_id=89)


@pytest.mark.parametrize("path", PATHS)
def test_longformer_dilation_two_heads_n4096(path):
    # dilation on two heads only (Longformer Tab. 12), causal, sampled rows
    H, n = 12, 4096
    dil = [0] * H
    dil[10], dil[11] = 2, 3
    gidx = torch.arange(16, dtype=torch.int32)
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([np.arange(0, 200), np.arange(n - 200, n), rng.choice(n, 300, replace=False)]))
    longformer_case(1, H, n, 64, 512, gidx, path=path, rows=rows, heads=[(0, 0), (0, 10), (0, 11)],
                    dilation=dil, causal=True, cfg_id=88)


@pytest.mark.parametrize("path", PATHS)
def test_bad_dilation_latches_status(path):
    Q, K, V = (t.cuda() for t in make_qkv(1, 2, 512, 64, "bf16", cfg_id=72))
    dil = torch.tensor([-1, 64], dtype=torch.int32).cuda()
    sa.set_option(sa.SA_OPT_FORCE_SIMT, 1 if path == "simt" else 0)
    try:
        sa.longformer_attn_fwd(Q, K, V, 64, None, dilation=dil)
        assert sa.get_last_device_status() == sa._lib.SA_ERR_BAD_INDEX
    finally:
        sa.set_option(sa.SA_OPT_FORCE_SIMT, 0)


# ------------------------------------------------------------- full-size workloads (sampled rows)

@pytest.mark.parametrize("path", PATHS)
def test_bigbird_n4096_workload(path):
    wl = WORKLOADS["bigbird_bf16_n4096"]
    rows = sampled_bigbird_rows(wl.n, wl.b, wl.g, seed=1)
    bigbird_case(wl.B, wl.H, wl.n, wl.d, wl.b, wl.g, wl.w, wl.r, cfg_id=wl.cfg_id, path=path,
                 rows=rows, heads=[(0, 0), (3, 7), (7, 11)])


def test_bigbird_n4096_workload_full_heads():
    # The headline workload through the tensor-core path in the bench's launch
    # configuration, two (batch, head) pairs compared on every row (all 64
    # query blocks: global tiles, window edges, every random block).
    wl = WORKLOADS["bigbird_bf16_n4096"]
    bigbird_case(wl.B, wl.H, wl.n, wl.d, wl.b, wl.g, wl.w, wl.r, cfg_id=wl.cfg_id, path="tc",
                 heads=[(2, 5), (6, 10)])


@pytest.mark.parametrize("path", PATHS)
def test_longformer_n4096_workload(path):
    wl = WORKLOADS["longformer_bf16_n4096"]
    gidx = torch.arange(wl.n_global, dtype=torch.int32)
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([np.arange(0, 300), np.arange(wl.n - 300, wl.n),
                                     rng.choice(wl.n, 600, replace=False)]))
    longformer_case(wl.B, wl.H, wl.n, wl.d, wl.window, gidx, cfg_id=wl.cfg_id, path=path, rows=rows,
                    heads=[(0, 0), (1, 5), (3, 11)])


@pytest.mark.parametrize("path", PATHS)
def test_bigbird_n16384_padded_workload(path):
    wl = WORKLOADS["bigbird_bf16_n16384_padded"]
    km = make_key_mask(wl.B, wl.n)
    rows = sampled_bigbird_rows(wl.n, wl.b, wl.g, seed=3)
    bigbird_case(wl.B, wl.H, wl.n, wl.d, wl.b, wl.g, wl.w, wl.r, cfg_id=wl.cfg_id, key_mask=km, path=path,
                 rows=rows, heads=[(0, 0), (1, 15)])


@pytest.mark.parametrize("path", PATHS)
def test_bigbird_n65536_d128_workload(path):
    wl = WORKLOADS["bigbird_bf16_n65536_d128"]
    rows = sampled_bigbird_rows(wl.n, wl.b, wl.g, n_random_blocks=4, seed=4)
    bigbird_case(wl.B, wl.H, wl.n, wl.d, wl.b, wl.g, wl.w, wl.r, sigma=wl.sigma, cfg_id=wl.cfg_id,
                 path=path, rows=rows, heads=[(0, 0), (0, 13)])


@pytest.mark.parametrize("path", PATHS)
def test_bigbird_etc_n4352_workload(path):
    """ETC bench shape (256 added global tokens + 4096, window 3 blocks, r = 0) against the ETC oracle."""
    from oracle import oracle_bigbird_etc
    from parity_util import assert_close
    wl = WORKLOADS["bigbird_etc_bf16_n4352"]
    Q, K, V = make_qkv(wl.B, wl.H, wl.n, wl.d, "bf16", cfg_id=wl.cfg_id)
    table = pattern_table(0, wl.H, wl.n, wl.b, wl.g, wl.w, wl.r)
    O = gpu_bigbird(Q, K, V, wl.b, wl.g, wl.w, wl.r, table, path=path).float().cpu()
    rows = sampled_bigbird_rows(wl.n, wl.b, wl.g, seed=6)
    for beta, h in [(0, 0), (7, 11)]:
        sl = (slice(beta, beta + 1), slice(h, h + 1))
        ref = oracle_bigbird_etc(Q[sl], K[sl], V[sl], wl.g * wl.b, wl.b, wl.w, rows=rows)[0, 0]
        assert_close(O[beta, h].numpy()[rows], ref, 2e-2, 2e-3, what=f"etc workload beta={beta} h={h}")


# ------------------------------------------------------------- properties

@pytest.mark.parametrize("path", PATHS)
def test_bigbird_deterministic(path):
    wl = WORKLOADS["bigbird_bf16_n4096"]
    Q, K, V = make_qkv(2, wl.H, wl.n, wl.d, "bf16", cfg_id=wl.cfg_id)
    table = pattern_table(0, wl.H, wl.n, wl.b, wl.g, wl.w, wl.r)
    O1 = gpu_bigbird(Q, K, V, wl.b, wl.g, wl.w, wl.r, table, path=path)
    O2 = gpu_bigbird(Q, K, V, wl.b, wl.g, wl.w, wl.r, table, path=path)
    assert torch.equal(O1, O2)


@pytest.mark.parametrize("path", PATHS)
def test_bad_random_index_latches_status(path):
    B, H, n, d, b, g, w, r = 1, 1, 512, 64, 64, 2, 3, 3
    Q, K, V = (t.cuda() for t in make_qkv(B, H, n, d, "bf16", cfg_id=70))
    table = pattern_table(0, H, n, b, g, w, r)
    table[0, 5, 1] = 1000  # out of [-1, nb): skipped by the kernel, latched as SA_ERR_BAD_INDEX
    sa.set_option(sa.SA_OPT_FORCE_SIMT, 1 if path == "simt" else 0)
    try:
        sa.bigbird_attn_fwd(Q, K, V, b, g, w, r, table.cuda())
        assert sa.get_last_device_status() == sa._lib.SA_ERR_BAD_INDEX
        assert sa.get_last_device_status() == 0  # reading clears it
    finally:
        sa.set_option(sa.SA_OPT_FORCE_SIMT, 0)


@pytest.mark.parametrize("path", PATHS)
def test_unsorted_global_index_latches_status(path):
    Q, K, V = (t.cuda() for t in make_qkv(1, 1, 512, 64, "bf16", cfg_id=71))
    gidx = torch.tensor([5, 3, 600], dtype=torch.int32).cuda()
    sa.set_option(sa.SA_OPT_FORCE_SIMT, 1 if path == "simt" else 0)
    try:
        sa.longformer_attn_fwd(Q, K, V, 64, gidx)
        assert sa.get_last_device_status() == sa._lib.SA_ERR_BAD_INDEX
    finally:
        sa.set_option(sa.SA_OPT_FORCE_SIMT, 0)


def test_tc_and_simt_agree_closely():
    wl = WORKLOADS["bigbird_bf16_n4096"]
    Q, K, V = make_qkv(1, 4, wl.n, wl.d, "bf16", cfg_id=72)
    table = pattern_table(0, 4, wl.n, wl.b, wl.g, wl.w, wl.r)
    a = gpu_bigbird(Q, K, V, wl.b, wl.g, wl.w, wl.r, table, path="tc").float()
    b = gpu_bigbird(Q, K, V, wl.b, wl.g, wl.w, wl.r, table, path="simt").float()
    assert (a - b).abs().max().item() <= 2e-2


def test_scratch_reuse_across_shapes():
    # Calls of different shapes share the library-owned scratch: split partials
    # of one call must not leak into the merge counters of the next.
    shapes = [(1, 2, 16384, 64, 64), (1, 2, 16384, 128, 128), (2, 2, 8192, 64, 64), (1, 3, 16384, 128, 128)]
    for (B, H, n, d, b) in shapes:
        rows = np.concatenate([np.arange(0, 2 * b), np.arange(n - b, n)])
        bigbird_case(B, H, n, d, b, 2, 3, 3, cfg_id=81, path="tc", rows=rows, heads=[(0, 0), (B - 1, H - 1)])


# ------------------------------------------------------ Longformer: separate global projections

def _gproj_case(B, H, n, d, window, gidx, path, key_mask=None, dilation=None, causal=False, rows=None, heads=None,
                cfg_id=90):
    from oracle import oracle_longformer
    from parity_util import assert_close, set_path

    Q, K, V = make_qkv(B, H, n, d, "bf16", cfg_id=cfg_id)
    Qg, Kg, Vg = make_qkv(B, H, n, d, "bf16", cfg_id=cfg_id + 1)
    dev = torch.device("cuda:0")
    set_path(path)
    try:
        O = sa.longformer_attn_fwd(*(t.to(dev) for t in (Q, K, V)), window, gidx.to(dev),
                                   None if key_mask is None else key_mask.to(dev),
                                   dilation=None if dilation is None else torch.tensor(dilation, dtype=torch.int32,
                                                                                       device=dev),
                                   causal=causal, Qg=Qg.to(dev), Kg=Kg.to(dev), Vg=Vg.to(dev))
        torch.cuda.synchronize()
        assert sa.get_last_device_status() == 0
    finally:
        set_path("tc")
    O = O.float().cpu()
    heads = heads if heads is not None else [(beta, h) for beta in range(B) for h in range(H)]
    for beta, h in heads:
        sl = (slice(beta, beta + 1), slice(h, h + 1))
        km = None if key_mask is None else key_mask[beta:beta + 1].numpy()
        ref = oracle_longformer(Q[sl], K[sl], V[sl], window, gidx.numpy(), key_mask=km, rows=rows,
                                dilation=None if dilation is None else [dilation[h]], causal=causal,
                                Qg=Qg[sl], Kg=Kg[sl], Vg=Vg[sl])[0, 0]
        got = O[beta, h].numpy() if rows is None else O[beta, h].numpy()[np.asarray(rows)]
        assert_close(got, ref, 2e-2, 2e-3, what=f"longformer gproj beta={beta} h={h}")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("d,dilation,causal", [(64, None, False), (64, [0, 2], True), (128, None, False)])
def test_longformer_global_projections_small(path, d, dilation, causal):
    B, n = 2, 1000
    _gproj_case(B, 2, n, d, 128, torch.tensor([0, 5, 500, 999], dtype=torch.int32), path,
                key_mask=make_key_mask(B, n), dilation=dilation, causal=causal)


@pytest.mark.parametrize("path", PATHS)
def test_longformer_global_projections_many_globals(path):
    """200 scattered global tokens: two global-row units per head, rows spread over all band tiles."""
    from block_sparse_long_bigbird_gb300.inputs import make_global_positions
    _gproj_case(1, 2, 3000, 64, 64, make_global_positions(3000, 200), path)


@pytest.mark.parametrize("path", PATHS)
def test_longformer_global_projections_bench_shape_sampled(path):
    """B=4 H=12 n=4096 window 512, globals 0..15: every global row and a band sample, two heads."""
    rows = np.concatenate([np.arange(0, 160), np.arange(2000, 2100), np.arange(4000, 4096)])
    _gproj_case(4, 12, 4096, 64, 512, torch.arange(16, dtype=torch.int32), path, rows=rows,
                heads=[(0, 0), (3, 11)])


# ------------------------------------------------------ BigBird-ETC through the ITC kernel

@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("g_tokens,b,n_reg", [(256, 64, 1024), (230, 64, 1024), (100, 128, 1024)])
def test_bigbird_etc_via_block_kernel(path, g_tokens, b, n_reg):
    """ETC (g added global tokens, window 3 blocks, r = 0): the global prefix is
    padded to whole blocks with tokens that key padding removes, then the
    block kernel runs with ceil(g / b) global blocks and no random blocks."""
    from oracle import oracle_bigbird_etc
    from parity_util import assert_close, gpu_bigbird
    B, H, d, w = 2, 2, 64, 3
    n = g_tokens + n_reg
    Q, K, V = make_qkv(B, H, n, d, "bf16", cfg_id=95)
    gb = -(-g_tokens // b)
    gp = gb * b
    padn = gp + n_reg
    pad = lambda x: torch.cat([x[:, :, :g_tokens], torch.zeros(B, H, gp - g_tokens, d, dtype=x.dtype),
                               x[:, :, g_tokens:]], dim=2).contiguous()
    km = torch.ones(B, padn, dtype=torch.uint8)
    km[:, g_tokens:gp] = 0
    table = pattern_table(0, H, padn, b, gb, w, 0)
    O = gpu_bigbird(pad(Q), pad(K), pad(V), b, gb, w, 0, table, km, path).float().cpu()
    keep = np.concatenate([np.arange(g_tokens), np.arange(gp, padn)])
    ref = oracle_bigbird_etc(Q, K, V, g_tokens, b, w)
    for beta in range(B):
        for h in range(H):
            assert_close(O[beta, h].numpy()[keep], ref[beta, h], 2e-2, 2e-3, what=f"etc beta={beta} h={h}")
    assert np.all(O[:, :, g_tokens:gp].numpy() == 0)


@pytest.mark.parametrize("path", PATHS)
def test_longformer_charlm_n23040_workload(path):
    """Autoregressive char-LM shape (B=16 H=8 n=23040, window 512, dilation 3 on
    the last two heads, causal, no global tokens): sampled rows of a plain and a
    dilated head, first and last batch entry."""
    wl = WORKLOADS["longformer_charlm_bf16_n23040"]
    rows = np.concatenate([np.arange(0, 300), np.arange(11000, 11500), np.arange(wl.n - 300, wl.n)])
    longformer_case(wl.B, wl.H, wl.n, wl.d, wl.window, None, cfg_id=wl.cfg_id, path=path, rows=rows,
                    heads=[(0, 0), (15, 7)], dilation=list(wl.dilation), causal=True)


@pytest.mark.parametrize("path", PATHS)
def test_longformer_gproj_n4096_workload(path):
    """Bench shape with separate global projections (generated as the bench does)."""
    wl = WORKLOADS["longformer_gproj_bf16_n4096"]
    rows = np.concatenate([np.arange(0, 200), np.arange(2000, 2100), np.arange(wl.n - 100, wl.n)])
    _gproj_case(wl.B, wl.H, wl.n, wl.d, wl.window, torch.arange(wl.n_global, dtype=torch.int32), path,
                rows=rows, heads=[(0, 0), (3, 11)], cfg_id=wl.cfg_id)


@pytest.mark.parametrize("chunk_keys,max_splits", [(0, 1), (512, 64), (2048, 16), (1 << 20, 16)])
def test_split_options_keep_the_result(chunk_keys, max_splits):
    # The split-KV chunking of the global tiles changes only the order in which
    # partial results are summed: every setting must match the oracle, the
    # global rows must stay within rounding of the default setting's, and the
    # local tiles must not change at all.
    B, H, n, d, b, g, w, r = 1, 2, 16384, 64, 64, 2, 3, 3
    Q, K, V = make_qkv(B, H, n, d, "bf16", cfg_id=140)
    table = pattern_table(0, H, n, b, g, w, r)
    km = make_key_mask(B, n, seed=23)
    base = gpu_bigbird(Q, K, V, b, g, w, r, table, km).float()
    sa.set_option(sa.SA_OPT_CHUNK_KEYS, chunk_keys)
    sa.set_option(sa.SA_OPT_MAX_SPLITS, max_splits)
    try:
        rows = sampled_bigbird_rows(n, b, g, n_random_blocks=3, seed=9)
        bigbird_case(B, H, n, d, b, g, w, r, cfg_id=140, key_mask=km, rows=rows, heads=[(0, 1)])
        O = gpu_bigbird(Q, K, V, b, g, w, r, table, km).float()
        longformer_case(1, 2, 12288, 64, 256, torch.arange(40, dtype=torch.int32), cfg_id=141,
                        rows=np.concatenate([np.arange(40), np.arange(5000, 5100)]))
    finally:
        sa.set_option(sa.SA_OPT_CHUNK_KEYS, 0)
        sa.set_option(sa.SA_OPT_MAX_SPLITS, 16)
    assert (O - base).abs().max().item() <= 2e-2
    assert torch.equal(O[:, :, g * b:], base[:, :, g * b:])


def test_dilated_heads_with_a_small_caller_workspace():
    # A caller-owned scratch sized by sa_longformer_workspace_bytes leaves no
    # room for the residue-class copies: the dilated heads then run over their
    # whole dilated reach. Both ways must match the oracle, and agree closely.
    B, H, n, d = 1, 4, 3000, 64
    dil = [0, 1, 2, 3]
    Q, K, V = make_qkv(B, H, n, d, "bf16", cfg_id=142)
    dev = torch.device("cuda:0")
    Qd, Kd, Vd = Q.to(dev), K.to(dev), V.to(dev)
    dt = torch.tensor(dil, dtype=torch.int32, device=dev)
    with_copies = sa.longformer_attn_fwd(Qd, Kd, Vd, 128, None, dilation=dt, causal=True)
    torch.cuda.synchronize()
    need = sa.longformer_workspace_bytes(B, H, n, d, 0)
    ws = torch.zeros((need + 255) // 256 * 256, dtype=torch.uint8, device=dev)
    sa.set_workspace(ws)
    try:
        without = sa.longformer_attn_fwd(Qd, Kd, Vd, 128, None, dilation=dt, causal=True)
        torch.cuda.synchronize()
        assert sa.get_last_device_status() == 0
    finally:
        sa.set_workspace(None)
    from oracle import oracle_longformer
    ref = oracle_longformer(Q, K, V, 128, np.zeros(0, np.int64), dilation=dil, causal=True)
    for O in (with_copies, without):
        err = np.abs(O.float().cpu().numpy() - ref)
        assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
    assert (with_copies.float() - without.float()).abs().max().item() <= 2e-2
    assert torch.equal(with_copies[:, 0], without[:, 0])  # dilation 0: the same kernel path
