"""The five synthetic workloads the library is measured and checked on.

BigBird-ITC shapes follow the paper's App. E Tab. 8 (block b = 64, g = 2b,
w = 3b, r = 3b tokens, i.e. 2 global, 3 window and 3 random blocks, n = 4096,
12 heads) and Longformer's Sec. 3.1 (window 512, i.e. 256 tokens each side,
global attention on a few chosen positions). The long and padded variants
stretch the same pattern to n = 16384 and n = 65536. The two ``*_bwd_*``
workloads time the backward (dQ, dK, dV) on the n = 4096 shapes. The ETC
workload adds 256 global tokens in front of 4096 regular ones (App. E: g = 256,
w = 3 blocks, r = 0), run as BigBird with 4 global blocks and no random blocks.
The char-LM workload follows Longformer's autoregressive setting (Sec. 4,
Tab. 12: 8 heads of 64, phase-5 sequences of 23,040 tokens, batch 16, window
512 in the bottom layer, dilation 3 on 2 heads in the top layers, no global
tokens). The gproj workload is the Longformer one with the separate
projections for global attention (Sec. 3.1).
"""

from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "bigbird" or "longformer"
    B: int
    H: int
    n: int
    d: int
    dtype: str           # "bf16" or "fp32"
    sigma: float = 1.0
    b: int = 64
    g: int = 2
    w: int = 3
    r: int = 3
    window: int = 0
    n_global: int = 0
    padded: bool = False
    seed: int = 0
    cfg_id: int = 0
    tol_max: float = 2e-2
    tol_mean: float = 2e-3
    grad: bool = False   # time the backward instead of the forward
    dilation: tuple = () # Longformer: per-head dilation (empty: 0 for every head)
    causal: bool = False # Longformer: autoregressive mode
    gproj: bool = False  # Longformer: separate projections for global attention


WORKLOADS = {
    "bigbird_fp32_n1024": Workload(
        "bigbird_fp32_n1024", "bigbird", B=1, H=1, n=1024, d=64, dtype="fp32",
        cfg_id=1, tol_max=1e-4, tol_mean=1e-5),
    "bigbird_bf16_n4096": Workload(
        "bigbird_bf16_n4096", "bigbird", B=8, H=12, n=4096, d=64, dtype="bf16", cfg_id=2),
    "longformer_bf16_n4096": Workload(
        "longformer_bf16_n4096", "longformer", B=4, H=12, n=4096, d=64, dtype="bf16",
        window=512, n_global=16, cfg_id=3),
    "bigbird_bf16_n16384_padded": Workload(
        "bigbird_bf16_n16384_padded", "bigbird", B=2, H=16, n=16384, d=64, dtype="bf16",
        padded=True, cfg_id=4),
    "bigbird_bf16_n65536_d128": Workload(
        "bigbird_bf16_n65536_d128", "bigbird", B=1, H=16, n=65536, d=128, dtype="bf16",
        sigma=0.5, b=128, cfg_id=5),
    "bigbird_etc_bf16_n4352": Workload(
        "bigbird_etc_bf16_n4352", "bigbird", B=8, H=12, n=4352, d=64, dtype="bf16", g=4, w=3, r=0, cfg_id=6),
    "longformer_charlm_bf16_n23040": Workload(
        "longformer_charlm_bf16_n23040", "longformer", B=16, H=8, n=23040, d=64, dtype="bf16",
        window=512, n_global=0, causal=True, dilation=(0, 0, 0, 0, 0, 0, 3, 3), cfg_id=7),
    "longformer_gproj_bf16_n4096": Workload(
        "longformer_gproj_bf16_n4096", "longformer", B=4, H=12, n=4096, d=64, dtype="bf16",
        window=512, n_global=16, gproj=True, cfg_id=3),
    "bigbird_bwd_bf16_n4096": Workload(
        "bigbird_bwd_bf16_n4096", "bigbird", B=8, H=12, n=4096, d=64, dtype="bf16", cfg_id=2, grad=True),
    "bigbird_bwd_bf16_n65536_d128": Workload(
        "bigbird_bwd_bf16_n65536_d128", "bigbird", B=1, H=16, n=65536, d=128, dtype="bf16",
        sigma=0.5, b=128, cfg_id=5, grad=True),
    "longformer_bwd_bf16_n4096": Workload(
        "longformer_bwd_bf16_n4096", "longformer", B=4, H=12, n=4096, d=64, dtype="bf16",
        window=512, n_global=16, cfg_id=3, grad=True),
}

HEADLINE = "bigbird_bf16_n4096"
