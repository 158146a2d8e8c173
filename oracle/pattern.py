"""BigBird random-block table, oracle side (test infrastructure, CPU only).

The BigBird paper (Sec. 2, Fig. 1a; App. E Tab. 8 "# of random token r = 3b")
and its blog summary (Sec. 2.1: each query attends r random keys; Sec. 4.2 (3):
the random blocks are gathered, r = 3) say only that every query block sees r
key blocks chosen at random. They name no generator. The table is therefore
pinned by a spec of our own, written out here in plain Python and implemented
independently in the C library:

* Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
  number generators", OOPSLA 2014), one sequential stream whose state starts
  at ``seed``.
* Visit order: heads h = 0..H-1, then query blocks j = g..nb-1. Global query
  blocks (j < g) attend every block already, draw nothing and hold -1.
* Candidates for block j: ascending list of key blocks kb in [0, nb) that are
  neither global (kb < g) nor in j's window (|kb - j| <= w // 2).
* Sampling: partial Fisher-Yates over the candidate list, k = min(r, m) draws;
  draw t picks index t + (u mod (m - t)) with u the next stream value.
* Output row: the k chosen blocks sorted ascending, then -1 up to r.
"""

import numpy as np

_MASK64 = (1 << 64) - 1
_GOLDEN_GAMMA = 0x9E3779B97F4A7C15


class SplitMix64:
    """SplitMix64 as published by Steele, Lea & Flood (OOPSLA 2014).

    The state advances by the golden-ratio increment; the output is the
    state passed through the variant-13 mix (shifts 30/27/31 with the two
    published odd multipliers). Arithmetic is modulo 2**64.
    """

    def __init__(self, seed):
        self.state = int(seed) & _MASK64

    def next(self):
        self.state = (self.state + _GOLDEN_GAMMA) & _MASK64
        z = self.state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
        return z ^ (z >> 31)


def splitmix64_stream(seed, count):
    """The first ``count`` outputs of SplitMix64 started at ``seed``."""
    gen = SplitMix64(seed)
    return [gen.next() for _ in range(count)]


def _candidates(nb, g, w, j):
    """Key blocks that block j may draw at random: not global, not in its window."""
    half = w // 2
    out = []
    for kb in range(nb):
        if kb < g:
            continue  # global column: already attended (blog Sec. 2.3)
        if abs(kb - j) <= half:
            continue  # window block: already attended (blog Sec. 2.2)
        out.append(kb)
    return out


def bigbird_random_table(seed, H, n, b, g, w, r):
    """int32 table [H, n // b, r] of random key blocks per (head, query block).

    Follows the spec in this module's docstring. The table depends only on
    (seed, H, n, b, g, w, r): it ignores key padding, and it is shared by every
    sequence of a batch.
    """
    if n % b != 0:
        raise ValueError("n must be a multiple of b")
    nb = n // b
    table = np.full((H, nb, r), -1, dtype=np.int32)
    gen = SplitMix64(seed)
    for h in range(H):
        for j in range(g, nb):
            cand = _candidates(nb, g, w, j)
            m = len(cand)
            k = min(r, m)
            for t in range(k):
                u = gen.next()
                idx = t + (u % (m - t))
                cand[t], cand[idx] = cand[idx], cand[t]
            chosen = sorted(cand[:k])
            for t, kb in enumerate(chosen):
                table[h, j, t] = kb
    return table
