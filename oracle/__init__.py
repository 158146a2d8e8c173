"""Oracle for sparse long-sequence attention: plain, slow, float64, CPU only.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline legs of ``bench.py`` may import this package. The product path (the
CUDA library under ``block_sparse_long_bigbird_gb300/``) never imports, links
or calls anything here, and nothing here imports the product package: the two
share no code. The seeded input generators live in their own module
(``block_sparse_long_bigbird_gb300/inputs.py``) and hold none of the method's
arithmetic.

Sources (web pages on block-sparse long-sequence attention):
  * "Big Bird: Transformers for Longer Sequences" (Zaheer et al.): the
    generalised attention Attn_D (Sec. 2, Eq. AT), the block-sparse
    implementation (App. D, Eq. 13, Fig. 6) and the ITC hyper-parameters
    (App. E, Tab. 8: g = 2b, w = 3b, r = 3b, b = 64).
  * The BigBird blog summary (Sec. 2.1-2.3, Sec. 4): random, window and global
    components restated where the paper's own Sec. 2 text is garbled.
  * "Longformer: The Long-Document Transformer" (Beltagy et al.): sliding
    window and symmetric global attention (Sec. 3.1), the dilated sliding
    window (Sec. 3.1, Fig. 2(c); per-head dilation, Tab. 12), the
    separate projections for global attention (Sec. 3.1), the
    autoregressive mode (App. B), scaled dot-product attention (Sec. 3.1,
    Eq. 1), and the slow per-diagonal "loop" variant used only for testing
    (Sec. 3.2, App. A), whose role this oracle plays.

Every function pinned by a test that does not reuse this code; the pins are in
``tests/test_oracle.py`` and ``tests/golden/``. Parity status per function:
  splitmix64_stream        pinned (published SplitMix64 test vector)
  bigbird_random_table     pinned (invariants, brute-force candidate sets,
                           sampling uniformity)
  bigbird_allowed          pinned (pure-Python enumeration, closed-form pair
                           counts, coverage => full attention)
  longformer_allowed       pinned (pure-Python enumeration, band/global
                           invariants, closed-form pair counts; dilation and
                           causal mode: enumeration of the window positions,
                           torch is_causal attention, per-residue-class full
                           attention, hand-derived pair counts)
  bigbird_etc_allowed,     pinned (pure-Python enumeration of the ETC rules;
  oracle_bigbird_etc       equals the ITC mask with g/b global blocks and r = 0
                           when b divides g; padded prefix equivalence)
  oracle_longformer with   pinned (global rows = torch SDPA of Qg, Kg, Vg over
  separate global          their keys; other rows identical to the single-
  projections              projection oracle; same tensors give the same result)
  masked_attention         pinned (torch float64 scaled_dot_product_attention
                           on full/block-diagonal/truncated cases, scalar-loop
                           brute force, single-key and row-sum identities)
  masked_attention_grads,  pinned (central finite differences of the pinned
  oracle_*_bwd             forward on tiny cases with padding, dilation and
                           causal mode; torch float64 autograd through
                           scaled_dot_product_attention with the same mask;
                           shift invariance sum_j dK_j = 0 and sum_j dV_j =
                           sum of dO over rows with an allowed key)
  oracle_bigbird_bwd_      pinned (equals the full oracle_bigbird_bwd at the
  sampled                  sampled rows and key blocks, with padding)
  masked_attention_grad_   pinned (brute-force sums of |term| and term^2 on
  terms                    a tiny case; the exact gradient lies inside the
                           rounding bound it yields for bf16-rounded P and dS)
"""

from .pattern import SplitMix64, splitmix64_stream, bigbird_random_table
from .attention import (
    bigbird_allowed,
    bigbird_etc_allowed,
    longformer_allowed,
    masked_attention,
    masked_softmax_probs,
    oracle_bigbird,
    oracle_bigbird_etc,
    oracle_longformer,
    masked_attention_grads,
    masked_attention_grad_terms,
    oracle_bigbird_bwd,
    oracle_bigbird_bwd_sampled,
    oracle_longformer_bwd,
    bigbird_attended_pairs,
    longformer_attended_pairs,
)

__all__ = [
    "SplitMix64",
    "splitmix64_stream",
    "bigbird_random_table",
    "bigbird_allowed",
    "bigbird_etc_allowed",
    "longformer_allowed",
    "masked_attention",
    "masked_softmax_probs",
    "oracle_bigbird",
    "oracle_bigbird_etc",
    "oracle_longformer",
    "masked_attention_grads",
    "masked_attention_grad_terms",
    "oracle_bigbird_bwd",
    "oracle_bigbird_bwd_sampled",
    "oracle_longformer_bwd",
    "bigbird_attended_pairs",
    "longformer_attended_pairs",
]
