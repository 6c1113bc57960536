"""Named synthetic MHLA workloads (shapes only, no arithmetic of the method).

Each workload fixes B, H, d, the token grid and the block shape, the input
dtype and how W is initialised.  The shapes stand in for the models the MHLA
pages evaluate (DeiT-T on 224 px, DiT-S/2 at 4096 px, SANA at 4096 px, a video
latent grid); no dataset or trained weight is involved.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from math import prod


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    d: int
    grid: tuple          # (Y, X) or (T, Y, X), raster order, last axis fastest
    block: tuple         # block extent per grid axis
    dtype: str           # "bf16" or "f32"
    transform: str       # W initialisation: linear | cos | exp | gaussian | local
    seed: int
    local_thres: float = 1.5
    exp_sigma: float = 3.0
    phi: str = "relu"    # relu | relu_eps
    eps: float = 1e-6
    note: str = field(default="", compare=False)

    @property
    def N(self) -> int:
        return prod(self.grid)

    @property
    def M(self) -> int:
        return prod(g // b for g, b in zip(self.grid, self.block))

    @property
    def w(self) -> int:
        return self.N // self.M

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    @property
    def tokens(self) -> int:
        """Tokens per forward pass (all heads of a token count once)."""
        return self.B * self.N

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes the pass must move at least: read q, k, v and write o."""
        return 4 * self.B * self.N * self.H * self.d * self.elem_bytes

    def describe(self) -> dict:
        return {
            "workload": self.name, "B": self.B, "H": self.H, "d": self.d,
            "N": self.N, "grid": list(self.grid), "block": list(self.block),
            "M": self.M, "dtype": self.dtype, "W_init": self.transform,
            "phi": self.phi, "eps": self.eps,
        }


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_16x16_fp32", 1, 1, 32, (16, 16), (4, 4), "f32", "linear", 1000,
                 note="16x16 grid, 4x4 blocks, fp32"),
        Workload("deit_t_14x14", 64, 3, 64, (14, 14), (2, 2), "bf16", "linear", 1001,
                 note="DeiT-T shaped: 196 tokens, 2x2 blocks (M=49)"),
        Workload("dit_s2_4096px", 4, 6, 64, (256, 256), (16, 16), "bf16", "exp", 1002,
                 note="DiT-S/2 at 4096 px: 65536 tokens, 16x16 blocks (M=256)"),
        Workload("sana_4096px", 2, 70, 32, (128, 128), (16, 16), "bf16", "linear", 1003,
                 note="SANA shaped 4096 px: 16384 tokens, d=32, 16x16 blocks (M=64)"),
        Workload("video_20x32x32", 2, 12, 64, (20, 32, 32), (4, 8, 8), "bf16", "linear", 1004,
                 note="video latent 20x32x32 (N=20480), 4x8x8 blocks (M=80)"),
    ]
    + [
        # causal language-model shape: a 1-D sequence of 4096 tokens in chunks of 64
        Workload("lm_causal_4096", 4, 12, 64, (1, 4096), (1, 64), "bf16", "linear", 1009,
                 note="causal sequence of 4096 tokens, 64-token blocks (M=64), 12 heads"),
    ]
    + [
        Workload(f"sweep_{s}x{s}", 4, 6, 64, (s, s), (16, 16), "bf16", "exp", 1005,
                 note=f"N sweep point {s}x{s} at 16x16 blocks")
        for s in (64, 128, 256, 512)
    ]
}

# The workload the headline throughput and HBM-roofline figures are quoted on.
HEADLINE = "dit_s2_4096px"
