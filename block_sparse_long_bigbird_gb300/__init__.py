"""GB300-native sparse long-sequence attention, forward and backward (BigBird-ITC and Longformer).

Python binding of the C ABI declared in ``include/sparse_attn.h``. The names
mirror the C entry points; the wrappers only marshal torch tensors (device
memory and the current CUDA stream) into pointers and sizes. All attention
arithmetic runs in the library's sm_103a kernels.
"""

import ctypes

import torch

from . import _lib
from ._lib import (  # noqa: F401
    SA_BF16,
    SA_FP32,
    SA_OPT_CHUNK_KEYS,
    SA_OPT_FORCE_SIMT,
    SA_OPT_GRID_CTAS,
    SA_OPT_MAX_SPLITS,
    SA_OPT_WAIT_LIMIT,
    SparseAttnError,
)

_DTYPE = {torch.bfloat16: SA_BF16, torch.float32: SA_FP32}


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check_qkv(Q, K, V):
    if Q.dtype not in _DTYPE:
        raise TypeError(f"unsupported dtype {Q.dtype}; use bfloat16 or float32")
    for t in (Q, K, V):
        if not t.is_cuda or t.dim() != 4 or not t.is_contiguous() or t.dtype != Q.dtype:
            raise ValueError("Q, K, V must be contiguous 4-D [B, H, n, d] CUDA tensors of one dtype")
        if t.shape != Q.shape or t.device != Q.device:
            raise ValueError("Q, K, V must share shape and device")


def build_bigbird_pattern(seed, H, n, b, g, w, r):
    """Per-head random key-block table, int32 CPU tensor [H, n // b, r]."""
    if b < 1 or n % b != 0:
        raise ValueError("n must be a positive multiple of b")
    out = torch.empty((H, n // b, r), dtype=torch.int32)
    _lib.check(_lib.lib().build_bigbird_pattern(ctypes.c_uint64(seed), H, n, b, g, w, r, _ptr(out)),
               "build_bigbird_pattern")
    return out


def bigbird_attn_fwd(Q, K, V, b, g, w, r, rand_idx, key_mask=None, out=None, stream=None):
    """BigBird-ITC block-sparse attention forward; returns O (same shape/dtype as Q).

    rand_idx: int32 CUDA tensor [H, n // b, r]; key_mask: uint8 CUDA tensor [B, n] or None.
    """
    _check_qkv(Q, K, V)
    B, H, n, d = Q.shape
    if out is None:
        out = torch.empty_like(Q)
    if rand_idx is not None and (not rand_idx.is_cuda or rand_idx.dtype != torch.int32
                                 or not rand_idx.is_contiguous()):
        raise ValueError("rand_idx must be a contiguous int32 CUDA tensor")
    if key_mask is not None and (not key_mask.is_cuda or key_mask.dtype != torch.uint8
                                 or not key_mask.is_contiguous()):
        raise ValueError("key_mask must be a contiguous uint8 CUDA tensor")
    st = _lib.lib().bigbird_attn_fwd(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(out), B, H, n, d, b, g, w, r,
        _ptr(rand_idx), _ptr(key_mask), _DTYPE[Q.dtype], _stream_handle(stream, Q.device))
    _lib.check(st, "bigbird_attn_fwd")
    return out


def longformer_attn_fwd(Q, K, V, window, global_idx, key_mask=None, out=None, stream=None, dilation=None,
                        causal=False, Qg=None, Kg=None, Vg=None):
    """Longformer sliding-window + global attention forward; returns O.

    global_idx: int32 CUDA tensor of sorted unique positions (may be empty or None).
    dilation: int32 CUDA tensor [H] of per-head dilations, or None (all 0).
    causal: autoregressive mode (no key after the query).
    Qg, Kg, Vg: the separate projections for global attention (all three or none):
    global rows are computed from them, every other row from Q, K, V.
    """
    _check_qkv(Q, K, V)
    B, H, n, d = Q.shape
    if out is None:
        out = torch.empty_like(Q)
    n_global = 0 if global_idx is None else int(global_idx.numel())
    if n_global and (not global_idx.is_cuda or global_idx.dtype != torch.int32
                     or not global_idx.is_contiguous()):
        raise ValueError("global_idx must be a contiguous int32 CUDA tensor")
    if key_mask is not None and (not key_mask.is_cuda or key_mask.dtype != torch.uint8
                                 or not key_mask.is_contiguous()):
        raise ValueError("key_mask must be a contiguous uint8 CUDA tensor")
    if dilation is not None and (not dilation.is_cuda or dilation.dtype != torch.int32
                                 or not dilation.is_contiguous() or dilation.numel() != H):
        raise ValueError("dilation must be a contiguous int32 CUDA tensor with one entry per head")
    sep = (Qg, Kg, Vg)
    if any(t is not None for t in sep):
        if any(t is None for t in sep):
            raise ValueError("pass all of Qg, Kg, Vg or none")
        _check_qkv(Qg, Kg, Vg)
        if Qg.shape != Q.shape or Qg.dtype != Q.dtype or Qg.device != Q.device:
            raise ValueError("Qg, Kg, Vg must match Q in shape, dtype and device")
    st = _lib.lib().longformer_attn_fwd_gproj(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(Qg), _ptr(Kg), _ptr(Vg), _ptr(out), B, H, n, d, window,
        _ptr(dilation), 1 if causal else 0, _ptr(global_idx if n_global else None), n_global, _ptr(key_mask),
        _DTYPE[Q.dtype], _stream_handle(stream, Q.device))
    _lib.check(st, "longformer_attn_fwd_gproj")
    return out


def _check_host(*tensors):
    for t in tensors:
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError("host entry points take contiguous CPU tensors (page-locked for overlapped copies)")


def bigbird_attn_fwd_host(Q, K, V, b, g, w, r, rand_idx, key_mask=None, out=None, stream=None, device=None):
    """bigbird_attn_fwd on CPU tensors (pinned for overlap); returns O as a CPU tensor.

    The copies are pipelined against the computation inside the library. The
    result is complete once `stream` (default: the current stream of `device`)
    has completed.
    """
    _check_host(Q, K, V, rand_idx, key_mask)
    if Q.dtype not in _DTYPE or K.shape != Q.shape or V.shape != Q.shape:
        raise ValueError("Q, K, V must share shape and a supported dtype")
    B, H, n, d = Q.shape
    if out is None:
        out = torch.empty(Q.shape, dtype=Q.dtype).pin_memory()
    _check_host(out)
    dev = device if device is not None else torch.cuda.current_device()
    st = _lib.lib().bigbird_attn_fwd_host(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(out), B, H, n, d, b, g, w, r,
        _ptr(rand_idx), _ptr(key_mask), _DTYPE[Q.dtype], _stream_handle(stream, dev))
    _lib.check(st, "bigbird_attn_fwd_host")
    return out


def longformer_attn_fwd_host(Q, K, V, window, global_idx, key_mask=None, out=None, stream=None, dilation=None,
                             causal=False, device=None):
    """longformer_attn_fwd on CPU tensors (pinned for overlap); returns O as a CPU tensor."""
    _check_host(Q, K, V, global_idx, key_mask, dilation)
    if Q.dtype not in _DTYPE or K.shape != Q.shape or V.shape != Q.shape:
        raise ValueError("Q, K, V must share shape and a supported dtype")
    B, H, n, d = Q.shape
    if out is None:
        out = torch.empty(Q.shape, dtype=Q.dtype).pin_memory()
    _check_host(out)
    n_global = 0 if global_idx is None else int(global_idx.numel())
    dev = device if device is not None else torch.cuda.current_device()
    st = _lib.lib().longformer_attn_fwd_host(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(out), B, H, n, d, window, _ptr(dilation), 1 if causal else 0,
        _ptr(global_idx if n_global else None), n_global, _ptr(key_mask), _DTYPE[Q.dtype],
        _stream_handle(stream, dev))
    _lib.check(st, "longformer_attn_fwd_host")
    return out


def _check_bwd(Q, K, V, dO):
    _check_qkv(Q, K, V)
    if not dO.is_cuda or not dO.is_contiguous() or dO.dtype != Q.dtype or dO.shape != Q.shape \
            or dO.device != Q.device:
        raise ValueError("dO must be a contiguous CUDA tensor shaped and typed like Q")


def _grad_outputs(Q, out):
    if out is None:
        return torch.empty_like(Q), torch.empty_like(Q), torch.empty_like(Q)
    dQ, dK, dV = out
    for t in (dQ, dK, dV):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != Q.dtype or t.shape != Q.shape:
            raise ValueError("gradient outputs must be contiguous CUDA tensors shaped and typed like Q")
    return dQ, dK, dV


def bigbird_attn_bwd(Q, K, V, dO, b, g, w, r, rand_idx, key_mask=None, out=None, stream=None):
    """Gradients (dQ, dK, dV) of bigbird_attn_fwd at (Q, K, V) for the upstream gradient dO.

    The pattern arguments are those of the forward call; out: optional (dQ, dK, dV) tensors.
    """
    _check_bwd(Q, K, V, dO)
    B, H, n, d = Q.shape
    dQ, dK, dV = _grad_outputs(Q, out)
    st = _lib.lib().bigbird_attn_bwd(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(dQ), _ptr(dK), _ptr(dV), B, H, n, d, b, g, w, r,
        _ptr(rand_idx), _ptr(key_mask), _DTYPE[Q.dtype], _stream_handle(stream, Q.device))
    _lib.check(st, "bigbird_attn_bwd")
    return dQ, dK, dV


def longformer_attn_bwd(Q, K, V, dO, window, global_idx, key_mask=None, dilation=None, causal=False,
                        out=None, stream=None):
    """Gradients (dQ, dK, dV) of longformer_attn_fwd at (Q, K, V) for the upstream gradient dO."""
    _check_bwd(Q, K, V, dO)
    B, H, n, d = Q.shape
    dQ, dK, dV = _grad_outputs(Q, out)
    n_global = 0 if global_idx is None else int(global_idx.numel())
    if dilation is not None and (not dilation.is_cuda or dilation.dtype != torch.int32
                                 or not dilation.is_contiguous() or dilation.numel() != H):
        raise ValueError("dilation must be a contiguous int32 CUDA tensor with one entry per head")
    st = _lib.lib().longformer_attn_bwd(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(dQ), _ptr(dK), _ptr(dV), B, H, n, d, window,
        _ptr(dilation), 1 if causal else 0, _ptr(global_idx if n_global else None), n_global, _ptr(key_mask),
        _DTYPE[Q.dtype], _stream_handle(stream, Q.device))
    _lib.check(st, "longformer_attn_bwd")
    return dQ, dK, dV


def longformer_attn_bwd_gproj(Q, K, V, Qg, Kg, Vg, dO, window, global_idx, key_mask=None, dilation=None,
                              causal=False, out=None, stream=None):
    """Gradients (dQ, dK, dV, dQg, dKg, dVg) of longformer_attn_fwd with separate global projections."""
    _check_bwd(Q, K, V, dO)
    _check_qkv(Qg, Kg, Vg)
    if Qg.shape != Q.shape or Qg.dtype != Q.dtype:
        raise ValueError("Qg, Kg, Vg must match Q in shape and dtype")
    B, H, n, d = Q.shape
    grads = out if out is not None else tuple(torch.empty_like(Q) for _ in range(6))
    n_global = 0 if global_idx is None else int(global_idx.numel())
    st = _lib.lib().longformer_attn_bwd_gproj(
        *(_ptr(t) for t in (Q, K, V, Qg, Kg, Vg, dO)), *(_ptr(t) for t in grads), B, H, n, d, window,
        _ptr(dilation), 1 if causal else 0, _ptr(global_idx if n_global else None), n_global, _ptr(key_mask),
        _DTYPE[Q.dtype], _stream_handle(stream, Q.device))
    _lib.check(st, "longformer_attn_bwd_gproj")
    return grads


def attn_bwd_workspace_bytes(B, H, n, d):
    return int(_lib.lib().sa_attn_bwd_workspace_bytes(B, H, n, d))


def get_last_device_status(stream=None, device=None):
    """Synchronise the stream and return (and clear) the latched device status code."""
    dev = device if device is not None else torch.cuda.current_device()
    return _lib.lib().sa_get_last_device_status(_stream_handle(stream, dev))


def check_wait_expiry(limit_us, stream=None, device=None):
    """Launch the failure-detection self-check: a bounded wait on a barrier that
    nothing arrives at, which must latch SA_ERR_TIMEOUT (read it with
    get_last_device_status)."""
    dev = device if device is not None else torch.cuda.current_device()
    _lib.check(_lib.lib().sa_check_wait_expiry(int(limit_us), _stream_handle(stream, dev)), "sa_check_wait_expiry")


def set_option(option, value):
    _lib.check(_lib.lib().sa_set_option(option, int(value)), "sa_set_option")


def bigbird_workspace_bytes(B, H, n, d, b, g):
    return int(_lib.lib().sa_bigbird_workspace_bytes(B, H, n, d, b, g))


def longformer_workspace_bytes(B, H, n, d, n_global):
    return int(_lib.lib().sa_longformer_workspace_bytes(B, H, n, d, n_global))


def set_workspace(tensor_or_none):
    """Use a caller-owned CUDA byte buffer as scratch (None: library-owned scratch)."""
    if tensor_or_none is None:
        _lib.check(_lib.lib().sa_set_workspace(ctypes.c_void_p(0), 0), "sa_set_workspace")
    else:
        t = tensor_or_none
        _lib.check(_lib.lib().sa_set_workspace(_ptr(t), t.numel() * t.element_size()), "sa_set_workspace")


def last_launch_count():
    return int(_lib.lib().sa_last_launch_count())
