"""Seeded synthetic inputs for the sparse-attention forward.

This module only draws random numbers and shapes tensors; it contains none of
the attention arithmetic, so the tests may feed the same inputs to the CUDA
library and to the float64 oracle.

Recipe (the pages publish no dataset for this kernel; BigBird App. E and the
Longformer paper Sec. 3 train on text that is out of scope here):
  * Q, K, V: ``torch.randn(B, H, n, d)`` in float32 from three CPU generators
    seeded ``1000 + 10 * cfg + {0, 1, 2}``, scaled by ``sigma``, then cast
    (round-to-nearest-even) to the working dtype.
  * Upstream gradient dO (backward): ``torch.randn(B, H, n, d)`` from a CPU
    generator seeded ``5000 + 10 * cfg``, cast like Q, K, V.
  * Key padding: per-sequence valid lengths ``L ~ U{n/2, ..., n}`` from a CPU
    generator seeded 2000; ``key_mask[beta, t] = t < L[beta]``.
  * BigBird random table: seed 0. The product draws it with
    ``build_bigbird_pattern``; the oracle side draws its own from the same
    spec, and the tests check that the two are bitwise equal.
"""

import torch

DTYPES = {"bf16": torch.bfloat16, "fp32": torch.float32}


def make_qkv(B, H, n, d, dtype="bf16", sigma=1.0, cfg_id=0):
    """Return CPU tensors (Q, K, V) of shape [B, H, n, d] in ``dtype``."""
    out = []
    for which in range(3):
        gen = torch.Generator(device="cpu")
        gen.manual_seed(1000 + 10 * cfg_id + which)
        x = torch.randn(B, H, n, d, generator=gen, dtype=torch.float32)
        if sigma != 1.0:
            x = x * sigma
        out.append(x.to(DTYPES[dtype]).contiguous())
    return tuple(out)


def make_grad_out(B, H, n, d, dtype="bf16", cfg_id=0):
    """Return a CPU tensor dO of shape [B, H, n, d] in ``dtype`` (upstream gradient)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(5000 + 10 * cfg_id)
    x = torch.randn(B, H, n, d, generator=gen, dtype=torch.float32)
    return x.to(DTYPES[dtype]).contiguous()


def make_lengths(B, n, seed=2000, low=None):
    """Valid lengths L[beta] uniform on {low, ..., n} (default low = n // 2)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    low = n // 2 if low is None else low
    return torch.randint(low, n + 1, (B,), generator=gen, dtype=torch.int64)


def make_key_mask(B, n, seed=2000, low=None):
    """uint8 [B, n] prefix mask, 1 = valid token, from ``make_lengths``."""
    lengths = make_lengths(B, n, seed=seed, low=low)
    t = torch.arange(n, dtype=torch.int64)
    return (t[None, :] < lengths[:, None]).to(torch.uint8).contiguous()


def make_random_key_mask(B, n, seed=3000, p_valid=0.8):
    """uint8 [B, n] mask with independent Bernoulli(p_valid) entries (edge tests)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    return (torch.rand(B, n, generator=gen) < p_valid).to(torch.uint8).contiguous()


def make_global_positions(n, count, seed=4000, first=False):
    """Sorted unique int32 token positions: the first ``count`` tokens when
    ``first`` is set, else ``count`` positions drawn without replacement."""
    if first:
        return torch.arange(count, dtype=torch.int32)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    perm = torch.randperm(n, generator=gen)[:count]
    return torch.sort(perm).values.to(torch.int32).contiguous()
