"""Host-only checks of the C ABI: exported symbols, the pattern builder and
argument validation. Nothing here launches a kernel or needs a GPU."""

import ctypes
import os
import re

import numpy as np
import pytest

from oracle import bigbird_random_table

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sparse_attn.h")


@pytest.fixture(scope="module")
def lib():
    from block_sparse_long_bigbird_gb300 import _build, _lib

    if not os.path.exists(_lib.LIB_PATH):
        _build.build()
    return _lib.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:sa_status|size_t|int|const char\s*\*)\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for required in ("build_bigbird_pattern", "bigbird_attn_fwd", "longformer_attn_fwd",
                     "sa_get_last_device_status", "sa_set_workspace"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from block_sparse_long_bigbird_gb300 import _lib

    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in sparse_attn.h but not exported"
        assert name in _lib.SIGNATURES, f"{name} has no ctypes signature"


@pytest.mark.parametrize("seed,H,n,b,g,w,r", [
    (0, 12, 4096, 64, 2, 3, 3),
    (0, 16, 65536, 128, 2, 3, 3),
    (0, 1, 1024, 64, 2, 3, 3),
    (12345, 3, 640, 64, 1, 5, 4),
    (7, 2, 256, 64, 0, 1, 9),
    (3, 1, 192, 64, 3, 3, 3),
    (2**64 - 1, 2, 2048, 128, 2, 7, 3),
])
def test_pattern_builder_bit_exact_vs_oracle(lib, seed, H, n, b, g, w, r):
    import block_sparse_long_bigbird_gb300 as sa

    got = sa.build_bigbird_pattern(seed, H, n, b, g, w, r).numpy()
    ref = bigbird_random_table(seed, H, n, b, g, w, r)
    assert got.dtype == np.int32 and got.shape == ref.shape
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("args", [
    (0, 0, 1024, 64, 2, 3, 3),     # H < 1
    (0, 1, 1000, 64, 2, 3, 3),     # n % b
    (0, 1, 1024, 64, -1, 3, 3),    # g < 0
    (0, 1, 1024, 64, 17, 3, 3),    # g > nb
    (0, 1, 1024, 64, 2, 4, 3),     # even w
    (0, 1, 1024, 64, 2, 3, -1),    # r < 0
])
def test_pattern_builder_rejects_bad_args(lib, args):
    buf = (ctypes.c_int32 * 64)()
    assert lib.build_bigbird_pattern(ctypes.c_uint64(args[0]), *args[1:], buf) == 1
    assert lib.build_bigbird_pattern(ctypes.c_uint64(0), 1, 1024, 64, 2, 3, 3, None) == 1


FAKE = 0x7f0000000000  # 256-byte aligned; never dereferenced: validation fails first


def _bb(lib, **kw):
    a = dict(Q=FAKE, K=FAKE + 0x100000, V=FAKE + 0x200000, O=FAKE + 0x300000, B=1, H=1, n=1024, d=64,
             b=64, g=2, w=3, r=3, rand=FAKE + 0x400000, km=None, dtype=0)
    a.update(kw)
    return lib.bigbird_attn_fwd(a["Q"], a["K"], a["V"], a["O"], a["B"], a["H"], a["n"], a["d"], a["b"],
                                a["g"], a["w"], a["r"], a["rand"], a["km"], a["dtype"], None)


@pytest.mark.parametrize("bad", [
    dict(Q=None), dict(O=None), dict(Q=FAKE + 8), dict(O=FAKE),
    dict(B=0), dict(H=0), dict(n=0), dict(d=96), dict(d=32), dict(b=32), dict(b=96),
    dict(n=1000), dict(g=-1), dict(g=17), dict(w=2), dict(w=0), dict(r=-1), dict(rand=None),
    dict(dtype=7),
])
def test_bigbird_invalid_args(lib, bad):
    assert _bb(lib, **bad) == 1


def _lf(lib, **kw):
    a = dict(Q=FAKE, K=FAKE + 0x100000, V=FAKE + 0x200000, O=FAKE + 0x300000, B=1, H=1, n=1024, d=64,
             window=64, gidx=FAKE + 0x400000, ng=4, km=None, dtype=0)
    a.update(kw)
    return lib.longformer_attn_fwd(a["Q"], a["K"], a["V"], a["O"], a["B"], a["H"], a["n"], a["d"],
                                   a["window"], a["gidx"], a["ng"], a["km"], a["dtype"], None)


@pytest.mark.parametrize("bad", [
    dict(K=None), dict(V=FAKE + 4), dict(B=-1), dict(d=100), dict(window=-2), dict(window=63),
    dict(ng=-1), dict(ng=1025), dict(gidx=None), dict(dtype=3),
])
def test_longformer_invalid_args(lib, bad):
    assert _lf(lib, **bad) == 1


def _lfx(lib, **kw):
    a = dict(Q=FAKE, K=FAKE + 0x100000, V=FAKE + 0x200000, O=FAKE + 0x300000, B=1, H=2, n=1024, d=64,
             window=64, dil=FAKE + 0x500000, causal=1, gidx=FAKE + 0x400000, ng=4, km=None, dtype=0)
    a.update(kw)
    return lib.longformer_attn_fwd_ex(a["Q"], a["K"], a["V"], a["O"], a["B"], a["H"], a["n"], a["d"],
                                      a["window"], a["dil"], a["causal"], a["gidx"], a["ng"], a["km"],
                                      a["dtype"], None)


@pytest.mark.parametrize("bad", [dict(causal=2), dict(causal=-1), dict(window=-2), dict(dtype=5), dict(V=None)])
def test_longformer_ex_invalid_args(lib, bad):
    assert _lfx(lib, **bad) == 1


def test_workspace_and_option_entry_points(lib):
    assert lib.sa_bigbird_workspace_bytes(1, 1, 1000, 64, 64, 2) == 0  # invalid sizes
    assert lib.sa_set_option(999, 1) == 1
    assert lib.sa_set_workspace(ctypes.c_void_p(FAKE + 16), 4096) == 1  # misaligned
    assert lib.sa_status_string(4) == b"SA_ERR_TIMEOUT"


def test_status_codes_match_header():
    from block_sparse_long_bigbird_gb300 import _lib

    text = open(HEADER).read()
    for name, val in [("SA_OK", _lib.SA_OK), ("SA_ERR_INVALID_ARG", _lib.SA_ERR_INVALID_ARG),
                      ("SA_ERR_UNSUPPORTED", _lib.SA_ERR_UNSUPPORTED), ("SA_ERR_CUDA", _lib.SA_ERR_CUDA),
                      ("SA_ERR_TIMEOUT", _lib.SA_ERR_TIMEOUT), ("SA_ERR_BAD_INDEX", _lib.SA_ERR_BAD_INDEX),
                      ("SA_BF16", _lib.SA_BF16), ("SA_FP32", _lib.SA_FP32)]:
        assert re.search(rf"\b{name}\s*=\s*{val}\b", text), name


def _bbb(lib, **kw):
    a = dict(Q=FAKE, K=FAKE + 0x100000, V=FAKE + 0x200000, dO=FAKE + 0x400000,
             dQ=FAKE + 0x500000, dK=FAKE + 0x600000, dV=FAKE + 0x700000, B=1, H=1, n=1024, d=64,
             b=64, g=2, w=3, r=3, rand=FAKE + 0x800000, km=None, dtype=0)
    a.update(kw)
    return lib.bigbird_attn_bwd(a["Q"], a["K"], a["V"], a["dO"], a["dQ"], a["dK"], a["dV"], a["B"],
                                a["H"], a["n"], a["d"], a["b"], a["g"], a["w"], a["r"], a["rand"], a["km"],
                                a["dtype"], None)


@pytest.mark.parametrize("bad", [
    dict(Q=None), dict(dO=None), dict(dQ=None), dict(dV=FAKE + 8), dict(dQ=FAKE), dict(dK=FAKE + 0x400000),
    dict(dV=FAKE + 0x500000), dict(n=1000), dict(d=32), dict(w=2), dict(r=-1), dict(rand=None), dict(dtype=2),
])
def test_bigbird_bwd_invalid_args(lib, bad):
    assert _bbb(lib, **bad) == 1


def _lfb(lib, **kw):
    a = dict(Q=FAKE, K=FAKE + 0x100000, V=FAKE + 0x200000, dO=FAKE + 0x400000,
             dQ=FAKE + 0x500000, dK=FAKE + 0x600000, dV=FAKE + 0x700000, B=1, H=2, n=1024, d=64,
             window=64, dil=None, causal=0, gidx=FAKE + 0x800000, ng=4, km=None, dtype=0)
    a.update(kw)
    return lib.longformer_attn_bwd(a["Q"], a["K"], a["V"], a["dO"], a["dQ"], a["dK"], a["dV"], a["B"],
                                   a["H"], a["n"], a["d"], a["window"], a["dil"], a["causal"], a["gidx"], a["ng"],
                                   a["km"], a["dtype"], None)


@pytest.mark.parametrize("bad", [
    dict(causal=2), dict(window=3), dict(ng=-1), dict(gidx=None), dict(dK=FAKE + 0x100000), dict(K=None),
    dict(d=100), dict(dtype=9),
])
def test_longformer_bwd_invalid_args(lib, bad):
    assert _lfb(lib, **bad) == 1


def test_bwd_workspace_bytes(lib):
    assert lib.sa_attn_bwd_workspace_bytes(8, 12, 4096, 64) == 2 * 4 * 8 * 12 * 4096
    assert lib.sa_attn_bwd_workspace_bytes(1, 2, 1000, 64) == 2 * 4 * 2 * 1024  # rows padded to 64
    assert lib.sa_attn_bwd_workspace_bytes(1, 1, 100, 96) == 0


def _lfg(lib, **kw):
    a = dict(Q=FAKE, K=FAKE + 0x100000, V=FAKE + 0x200000, Qg=FAKE + 0x500000, Kg=FAKE + 0x600000,
             Vg=FAKE + 0x700000, O=FAKE + 0x300000, B=1, H=2, n=1024, d=64, window=64, dil=None, causal=0,
             gidx=FAKE + 0x400000, ng=4, km=None, dtype=0)
    a.update(kw)
    return lib.longformer_attn_fwd_gproj(a["Q"], a["K"], a["V"], a["Qg"], a["Kg"], a["Vg"], a["O"], a["B"], a["H"],
                                         a["n"], a["d"], a["window"], a["dil"], a["causal"], a["gidx"], a["ng"],
                                         a["km"], a["dtype"], None)


@pytest.mark.parametrize("bad", [dict(Kg=None), dict(Qg=None, Kg=None), dict(Vg=FAKE + 8), dict(O=FAKE + 0x500000),
                                 dict(causal=3), dict(window=5)])
def test_longformer_gproj_invalid_args(lib, bad):
    assert _lfg(lib, **bad) == 1


def test_split_options_shape_the_workspace(lib):
    from block_sparse_long_bigbird_gb300 import _lib

    # A global tile's sweep is cut into split-KV chunks only when it is long
    # against the call's other work; SA_OPT_CHUNK_KEYS forces a chunk length
    # and SA_OPT_MAX_SPLITS bounds the count. The scratch need follows (host
    # arithmetic only, no device).
    args = (1, 2, 16384, 64, 64, 2)  # few heads: long global sweeps, split by default
    base = lib.sa_bigbird_workspace_bytes(*args)
    big = lib.sa_bigbird_workspace_bytes(8, 12, 4096, 64, 64, 2)  # upper bound over w, r
    try:
        assert lib.sa_set_option(_lib.SA_OPT_MAX_SPLITS, 1) == _lib.SA_OK
        one = lib.sa_bigbird_workspace_bytes(*args)
        assert one < base  # no partials
        assert lib.sa_set_option(_lib.SA_OPT_MAX_SPLITS, 16) == _lib.SA_OK
        assert lib.sa_set_option(_lib.SA_OPT_CHUNK_KEYS, 1 << 20) == _lib.SA_OK
        assert lib.sa_bigbird_workspace_bytes(*args) == one  # one chunk covers every key
        assert lib.sa_set_option(_lib.SA_OPT_CHUNK_KEYS, 512) == _lib.SA_OK
        assert lib.sa_bigbird_workspace_bytes(*args) >= base  # 16 chunks of 8 steps at most
        assert lib.sa_set_option(_lib.SA_OPT_CHUNK_KEYS, -5) == _lib.SA_OK  # back to the default
        assert lib.sa_bigbird_workspace_bytes(*args) == base
        assert lib.sa_bigbird_workspace_bytes(8, 12, 4096, 64, 64, 2) == big
    finally:
        lib.sa_set_option(_lib.SA_OPT_CHUNK_KEYS, 0)
        lib.sa_set_option(_lib.SA_OPT_MAX_SPLITS, 16)
