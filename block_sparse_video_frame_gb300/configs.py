"""Workload presets: the five attention shapes this library is measured and tested on.

Each preset is plain data (sizes, window, reference frame, how the synthetic
inputs are drawn). Nothing here computes any part of the attention method.

Shapes follow the super-resolution and base-DiT attention described in
"HeyGen x Google Cloud: Bringing Avatar IV to TPUs" ("Deleting the Mask":
a query attends to the frames within W of its own frame and to one fixed
reference frame; 720p/1080p output from "The Workload, and the Port"). The token counts
per frame are latent patch grids (20x20, 45x80, 68x120, 30x52).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Tuple


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    D: int
    F: int             # frames in the sequence
    T: int             # tokens per frame
    W: int             # window radius in frames (W >= F-1 means dense)
    ref: int           # global reference frame index, -1 for none
    block_size: int    # schedule block size: multiple of 16 dividing T (dense: any multiple of 16)
    key_offset_scale: float = 0.5          # per-head key mean offset drawn as s * N(0, 1)^D
    outlier_heads: Tuple[int, ...] = ()    # heads given one key scaled x20
    seed: int = 0
    extra: dict = field(default_factory=dict, compare=False)

    @property
    def N(self) -> int:
        return self.F * self.T

    @property
    def scale(self) -> float:
        return 1.0 / float(self.D) ** 0.5

    @property
    def dense(self) -> bool:
        return self.W >= self.F - 1

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


TINY = Workload("tiny", B=1, H=2, D=64, F=4, T=48, W=1, ref=0, block_size=16,
                outlier_heads=(1,), seed=0)
SMALL = Workload("small", B=1, H=8, D=128, F=9, T=400, W=1, ref=0, block_size=80,
                 outlier_heads=(7,), seed=1)
SR720 = Workload("sr720p", B=1, H=24, D=128, F=13, T=3600, W=2, ref=0, block_size=240,
                 outlier_heads=(23,), seed=2)
SR1080 = Workload("sr1080p", B=1, H=24, D=128, F=9, T=8160, W=1, ref=0, block_size=240,
                  outlier_heads=(), seed=3)
DENSE = Workload("dense_base", B=1, H=24, D=128, F=21, T=1560, W=20, ref=0, block_size=16,
                 outlier_heads=(18, 19, 20, 21, 22, 23), seed=4)

ALL = (TINY, SMALL, SR720, SR1080, DENSE)
# 720p-like geometry with 8 heads (Q+K+V = 288 MB, still larger than L2): the
# case profiled with the full ncu section set.
SR720_H8 = SR720.with_(name="sr720p_h8", H=8, outlier_heads=(7,))
# the same hidden size split into 48 heads of 64 (the D = 64 kernel at scale)
SR720_D64 = SR720.with_(name="sr720p_d64", D=64, H=48, outlier_heads=(47,))
# 16 heads of 64: the bytes and FLOPs of sr720p_h8 at the other head dim (profiling size)
SR720_D64_H16 = SR720.with_(name="sr720p_d64_h16", D=64, H=16, outlier_heads=(15,))
BY_NAME = {w.name: w for w in ALL + (SR720_H8, SR720_D64, SR720_D64_H16)}


def dense_sweep():
    """The dense base-DiT eligibility sweep: key offset scale s in {0, 0.5, 2}
    crossed with 0, 1 and 6 of 24 outlier heads (0-25%)."""
    out = []
    for s in (0.0, 0.5, 2.0):
        for n_out in (0, 1, 6):
            heads = tuple(range(DENSE.H - n_out, DENSE.H))
            out.append(DENSE.with_(name=f"dense_s{s:g}_out{n_out}", key_offset_scale=s,
                                   outlier_heads=heads))
    return out


@dataclass(frozen=True)
class PrologueShape:
    """Sizes of the fused pre-attention chain ("Layout Is the ABI"): B x N
    token rows of hidden size C projected to H heads of size D for q, k, v."""
    name: str
    B: int
    N: int
    C: int
    H: int
    D: int
    eps: float = 1e-6
    base: float = 10000.0
    seed: int = 0

    @property
    def O(self) -> int:
        return 3 * self.H * self.D

    @property
    def flops(self) -> int:
        """Dense projection FLOPs (2 per multiply-add)."""
        return 2 * self.B * self.N * self.C * self.O


# Hidden size = H * D (the attention width of the shapes above).
PRO_TINY = PrologueShape("pro_tiny", B=1, N=200, C=128, H=2, D=64)           # ragged rows, one column tile
PRO_RAGGED = PrologueShape("pro_ragged", B=2, N=300, C=200, H=3, D=128, seed=1)  # K tail, half column tile
PRO_SMALL = PrologueShape("pro_small", B=1, N=3600, C=1024, H=8, D=128, seed=2)
PRO_SR720 = PrologueShape("pro_sr720p", B=1, N=46800, C=3072, H=24, D=128, seed=3)
# W' of 35 MB: the GEMM walks its column tiles in two bands (23 tiles: 12 + 11, the
# last one half wide) over 700 ragged rows
PRO_BANDS = PrologueShape("pro_bands", B=1, N=700, C=3072, H=15, D=128, seed=4)
PROLOGUE = (PRO_TINY, PRO_RAGGED, PRO_SMALL, PRO_SR720)
