"""Seeded synthetic workloads: block layouts and Q/K/V tensors.

This module holds input generation only and none of the attention arithmetic; the
tests, the benchmark and the oracle checks all draw their inputs from it.

The five workloads (batch B, heads H, sequence L, block b, head dim d):

  1 ``tiny-band1``        1,  2,   256,  64,  64  band |i-j| <= 1 on a 4x4 grid, fp32 source
  2 ``band4``             1,  8,  4096,  64,  64  band |i-j| <= 4 (the local pattern of the
                                                  DeepSpeed utils page's usage example)
  3 ``window4-global0``   2, 16,  8192, 128, 128  j in [i-3, i] plus column 0, causal diagonal
  4 ``bernoulli0.1``      4, 16, 16384,  64, 128  per-head tril(Bernoulli(0.10), -1) | eye,
                                                  causal diagonal
  5 ``strided16-band8``   1, 32, 65536, 128, 128  j in [i-7, i] or (j % 16 == 15 and j <= i),
                                                  causal diagonal (Sparse-Transformer style)

Recipe: Q, K, V are drawn in that order with ``torch.randn(B, H, L, d,
generator=g)`` in fp32 on the CPU, ``g.manual_seed(1234 + index)``, and rounded to
bf16 (round-to-nearest-even).  Workload 4 draws head h's layout from its own
generator seeded ``1000 + h``: ``keep = torch.rand(nb, nb) < 0.10``.
"""

from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    index: int
    name: str
    B: int
    H: int
    L: int
    block: int
    d: int
    causal_diag: bool

    @property
    def nb(self) -> int:
        return self.L // self.block

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def describe(self) -> str:
        return (f"{self.name}: B={self.B} H={self.H} L={self.L} block={self.block} "
                f"d={self.d} causal_diag={int(self.causal_diag)}")


WORKLOADS = {
    1: Workload(1, "tiny-band1", 1, 2, 256, 64, 64, False),
    2: Workload(2, "band4", 1, 8, 4096, 64, 64, False),
    3: Workload(3, "window4-global0", 2, 16, 8192, 128, 128, True),
    4: Workload(4, "bernoulli0.1", 4, 16, 16384, 64, 128, True),
    5: Workload(5, "strided16-band8", 1, 32, 65536, 128, 128, True),
}


# ------------------------------------------------------------------ layout builders


def band_layout(H: int, nb: int, w: int) -> torch.Tensor:
    """Local band |i - j| <= w for every head."""
    i = torch.arange(nb)[:, None]
    j = torch.arange(nb)[None, :]
    lay = ((i - j).abs() <= w).to(torch.int32)
    return lay.expand(H, nb, nb).contiguous()


def window_global_layout(H: int, nb: int, w: int = 3) -> torch.Tensor:
    """Block-causal window j in [i - w, i] plus global column 0."""
    i = torch.arange(nb)[:, None]
    j = torch.arange(nb)[None, :]
    lay = (((j <= i) & (j >= i - w)) | (j == 0)).to(torch.int32)
    return lay.expand(H, nb, nb).contiguous()


def bernoulli_causal_layout(H: int, nb: int, p: float = 0.10, seed0: int = 1000) -> torch.Tensor:
    """Per head h: strictly-lower blocks kept i.i.d. with probability p (seed seed0 + h),
    diagonal always kept."""
    out = torch.empty(H, nb, nb, dtype=torch.int32)
    eye = torch.eye(nb, dtype=torch.bool)
    for h in range(H):
        g = torch.Generator().manual_seed(seed0 + h)
        keep = torch.rand(nb, nb, generator=g) < p
        out[h] = (torch.tril(keep, -1) | eye).to(torch.int32)
    return out


def strided_layout(H: int, nb: int, w: int = 7, stride: int = 16) -> torch.Tensor:
    """Sparse-Transformer style: band j in [i - w, i] plus columns j % stride == stride - 1, j <= i."""
    i = torch.arange(nb)[:, None]
    j = torch.arange(nb)[None, :]
    lay = (((j <= i) & (j >= i - w)) | ((j % stride == stride - 1) & (j <= i))).to(torch.int32)
    return lay.expand(H, nb, nb).contiguous()


def layout_for(wl: Workload) -> torch.Tensor:
    """The int32 [H, nb, nb] layout of a workload."""
    if wl.index == 1:
        return band_layout(wl.H, wl.nb, 1)
    if wl.index == 2:
        return band_layout(wl.H, wl.nb, 4)
    if wl.index == 3:
        return window_global_layout(wl.H, wl.nb, 3)
    if wl.index == 4:
        return bernoulli_causal_layout(wl.H, wl.nb)
    if wl.index == 5:
        return strided_layout(wl.H, wl.nb)
    raise KeyError(wl.index)


def random_layout(H: int, nb: int, p: float, seed: int, empty_rows: int = 0) -> torch.Tensor:
    """Random 0/1 layout for tests; optionally forces ``empty_rows`` all-zero rows per head."""
    g = torch.Generator().manual_seed(seed)
    lay = (torch.rand(H, nb, nb, generator=g) < p).to(torch.int32)
    for h in range(H):
        if empty_rows:
            rows = torch.randperm(nb, generator=g)[:empty_rows]
            lay[h, rows] = 0
    return lay


# ---------------------------------------------------------------------- tensors


def qkv(wl: Workload, seed: int | None = None, dtype=torch.bfloat16, B: int | None = None,
        H: int | None = None, L: int | None = None):
    """Q, K, V on the CPU, drawn in that order from one generator, rounded to ``dtype``.

    ``B``/``H``/``L`` override the workload's sizes (smaller test cases)."""
    B = wl.B if B is None else B
    H = wl.H if H is None else H
    L = wl.L if L is None else L
    g = torch.Generator().manual_seed(1234 + wl.index if seed is None else seed)
    out = []
    for _ in range(3):
        t = torch.randn(B, H, L, wl.d, generator=g, dtype=torch.float32)
        out.append(t.to(dtype))
    return tuple(out)


def randn_qkv(B: int, H: int, L: int, d: int, seed: int, dtype=torch.bfloat16):
    """Q, K, V ~ N(0, 1) of an arbitrary shape (tests)."""
    g = torch.Generator().manual_seed(seed)
    return tuple(torch.randn(B, H, L, d, generator=g).to(dtype) for _ in range(3))


# ------------------------------------------------------- top-k token-gather workload


@dataclasses.dataclass(frozen=True)
class TopkWorkload:
    """Top-k token-gather attention (the DeepSeek-V4.1 sparse_attn shape: 64 heads of
    512, one key-value row shared by all heads): M query positions at the end of an
    N-row context, each listing K rows."""
    name: str
    B: int
    M: int
    N: int
    H: int
    D: int
    K: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


TOPK = TopkWorkload("topk2048-ctx65536", 1, 4096, 65536, 64, 512, 2048)


def topk_inputs(B: int, M: int, N: int, H: int, D: int, K: int, seed: int):
    """q [B, M, H, D], kv [B, N, D] ~ N(0, 1) rounded to bf16; sink [H] ~ N(0, 1) fp32;
    idx int32 [B, M, K].

    Position m stands at N - M + m and may list rows 0 .. N - M + m (causal).  Its K
    rows are drawn one per stratum of that range (row floor((j + u_j) * count / K) for
    j < K, u_j uniform in [0, 1)), so they are distinct, ascending and spread over the
    whole context; a position with fewer than K candidates lists them all and pads with -1.
    """
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, M, H, D, generator=g).to(torch.bfloat16)
    kv = torch.randn(B, N, D, generator=g).to(torch.bfloat16)
    sink = torch.randn(H, generator=g)
    count = (N - M + torch.arange(M) + 1).clamp(min=1)           # candidates per position
    u = torch.rand(B, M, K, generator=g, dtype=torch.float64)
    j = torch.arange(K, dtype=torch.float64)
    idx = torch.floor((j + u) * count[None, :, None].double() / K).to(torch.int64)
    short = count[None, :, None] < K                                 # fewer candidates than K
    idx = torch.where(short, torch.where(j[None, None, :] < count[None, :, None],
                                         j.to(torch.int64)[None, None, :].expand(B, M, K), -1), idx)
    return q, kv, sink, idx.to(torch.int32)
