"""Failure detection and the scratch-sharing contract, on the GPU, without a
fault: a wait is made to run out (a barrier nothing arrives at, through the
kernels' own bounded-wait helper; and a very short pipeline limit on a real
call), and the device must end with SA_ERR_TIMEOUT latched, or nothing
latched, and a usable context whose next call is exact.

The pages define no such path; it belongs to the library's boundary (bounded
waits, a latched device status word, scratch shared by the calls of a device).
"""

import numpy as np
import pytest
import torch

import block_sparse_long_bigbird_gb300 as sa
from block_sparse_long_bigbird_gb300 import _lib
from block_sparse_long_bigbird_gb300.inputs import make_key_mask, make_qkv
from oracle import oracle_bigbird
from parity_util import assert_close, pattern_table, sampled_bigbird_rows


def _check_rows(O, Q, K, V, b, g, w, table, km, heads, rows):
    for beta, h in heads:
        sl = (slice(beta, beta + 1), slice(h, h + 1))
        kmb = None if km is None else km[beta:beta + 1].numpy()
        ref = oracle_bigbird(Q[sl], K[sl], V[sl], b, g, w, table.numpy()[h:h + 1], key_mask=kmb, rows=rows)[0, 0]
        assert_close(O[beta, h].float().cpu().numpy()[rows], ref, 2e-2, 2e-3, what=f"beta={beta} h={h}")


@pytest.mark.gpu
def test_wait_limit_expiry_is_clean_and_the_next_call_is_exact():
    # n = 16384 splits the global tiles, so an aborted call can leave split-merge
    # counters set; the next call runs WITHOUT reading the status in between,
    # so it must find the scratch clean by itself.
    B, H, n, d, b, g, w, r = 1, 4, 16384, 64, 64, 2, 3, 3
    dev = torch.device("cuda:0")
    Qc, Kc, Vc = make_qkv(B, H, n, d, "bf16", cfg_id=120)
    Q, K, V = Qc.to(dev), Kc.to(dev), Vc.to(dev)
    table = pattern_table(0, H, n, b, g, w, r)
    tab = table.to(dev)
    km = make_key_mask(B, n, seed=21)
    kmd = km.to(dev)
    assert sa.get_last_device_status() == 0
    sa.set_option(sa.SA_OPT_WAIT_LIMIT, 1)  # 1 microsecond: waits on copies and MMAs run out
    try:
        for _ in range(3):
            sa.bigbird_attn_fwd(Q, K, V, b, g, w, r, tab, kmd)
        torch.cuda.synchronize()  # the kernels end by themselves: every wait and every drain is bounded
    finally:
        sa.set_option(sa.SA_OPT_WAIT_LIMIT, 0)  # back to the default
    O = sa.bigbird_attn_fwd(Q, K, V, b, g, w, r, tab, kmd)
    torch.cuda.synchronize()
    st = sa.get_last_device_status()
    assert st in (_lib.SA_OK, _lib.SA_ERR_TIMEOUT), _lib.STATUS_NAMES.get(st, st)
    assert sa.get_last_device_status() == 0  # reading clears it
    rows = sampled_bigbird_rows(n, b, g, n_random_blocks=4, seed=3)
    _check_rows(O, Qc, Kc, Vc, b, g, w, table, km, [(0, 0), (0, 3)], rows)
    # and once more after the status read (which re-zeroes the scratch)
    O2 = sa.bigbird_attn_fwd(Q, K, V, b, g, w, r, tab, kmd)
    torch.cuda.synchronize()
    assert sa.get_last_device_status() == 0
    assert torch.equal(O, O2)


@pytest.mark.gpu
def test_expired_wait_latches_timeout_and_the_context_stays_usable():
    # The self-check waits, through the kernels' own bounded-wait helper, on a
    # barrier that nothing arrives at: the wait must give up and latch
    # SA_ERR_TIMEOUT, and an ordinary call afterwards must be exact.
    assert sa.get_last_device_status() == 0
    sa.check_wait_expiry(2000)  # 2 ms
    assert sa.get_last_device_status() == _lib.SA_ERR_TIMEOUT
    assert sa.get_last_device_status() == 0  # reading clears it
    B, H, n, d, b, g, w, r = 2, 2, 2048, 64, 64, 2, 3, 3
    Q, K, V = make_qkv(B, H, n, d, "bf16", cfg_id=122)
    table = pattern_table(0, H, n, b, g, w, r)
    dev = torch.device("cuda:0")
    O = sa.bigbird_attn_fwd(Q.to(dev), K.to(dev), V.to(dev), b, g, w, r, table.to(dev))
    torch.cuda.synchronize()
    assert sa.get_last_device_status() == 0
    _check_rows(O, Q, K, V, b, g, w, table, None, [(0, 0), (1, 1)], np.arange(n))


def test_wait_expiry_self_check_rejects_bad_limits():
    lib = _lib.lib()
    assert lib.sa_check_wait_expiry(0, None) == _lib.SA_ERR_INVALID_ARG
    assert lib.sa_check_wait_expiry(2000001, None) == _lib.SA_ERR_INVALID_ARG


@pytest.mark.gpu
def test_calls_on_two_event_ordered_streams_share_the_scratch():
    # The scratch is per device: calls on two streams are safe when the
    # streams are ordered. Each call's output must equal the same call made
    # alone on the default stream (bitwise: the kernel is deterministic).
    dev = torch.device("cuda:0")
    shapes = [(1, 2, 16384, 64, 64), (2, 4, 4096, 64, 64), (1, 2, 8192, 128, 128)]
    probs = []
    for i, (B, H, n, d, b) in enumerate(shapes):
        Q, K, V = (t.to(dev) for t in make_qkv(B, H, n, d, "bf16", cfg_id=130 + i))
        tab = pattern_table(0, H, n, b, 2, 3, 3).to(dev)
        probs.append((Q, K, V, b, tab))
    alone = []
    for Q, K, V, b, tab in probs:
        alone.append(sa.bigbird_attn_fwd(Q, K, V, b, 2, 3, 3, tab))
    torch.cuda.synchronize()
    assert sa.get_last_device_status() == 0
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    outs = []
    prev = torch.cuda.current_stream(dev)
    for k, (Q, K, V, b, tab) in enumerate(probs * 2):
        s = s1 if k % 2 == 0 else s2
        s.wait_stream(prev)  # order this call after the previous one
        with torch.cuda.stream(s):
            outs.append(sa.bigbird_attn_fwd(Q, K, V, b, 2, 3, 3, tab, stream=s))
        prev = s
    torch.cuda.synchronize()
    assert sa.get_last_device_status() == 0
    for k, o in enumerate(outs):
        assert torch.equal(o, alone[k % len(probs)]), f"call {k} differs from the same call made alone"
    assert np.isfinite(outs[0].float().cpu().numpy()).all()
