"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers; it contains none of the attention
arithmetic.  The same bytes feed the CUDA library and the fp64 oracle.

Recipe: a CPU ``torch.Generator`` seeded with ``seed`` draws, in this order,
Q, K, V (and dO when the workload has a backward pass) as fp32 standard
normals of shape [B, H, N, d], each multiplied by ``value_scale``.  When
``outlier_frac`` > 0, for every (b, h) a set of round(outlier_frac * N) query
rows and, independently, a set of key rows (both from ``torch.randperm`` on
the same generator, Q first) are multiplied by ``outlier_mult``.  When
``entry_outlier_frac`` > 0, Q, K and V in turn draw a uniform [0, 1) tensor
and a standard normal tensor of their shape; the entries whose uniform is
below ``entry_outlier_frac`` are replaced by that normal times
``entry_outlier_std`` (isolated large entries, the kind of outlier that
block scales handle worst).  Finally every tensor is rounded to bf16
(round-to-nearest-even, torch ``.to``).

``make_inputs_device`` draws the same recipe (without outlier rows) with a
generator on the GPU, for shapes too large to draw on the host: Q, K, V
(and dO) in that order, each a standard normal tensor in fp32 times
``value_scale``, rounded to bf16.  Its bytes differ from ``make_inputs``'s
(another generator); the oracle is given slices of the same tensors.

``random_signs`` draws the +-1 diagonal of the random orthogonal matrix used
for incoherent processing before FP8 quantization.
"""

from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    value_scale: float = 1.0
    outlier_frac: float = 0.0
    outlier_mult: float = 1.0
    backward: bool = True
    seed: int = 1000
    check_rows: int = 0          # >0: the oracle checks this many rows per head
    entry_outlier_frac: float = 0.0
    entry_outlier_std: float = 1.0

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(d), rounded to fp32 (the kernels' type)."""
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32))

    def with_n(self, n: int) -> "Workload":
        return dataclasses.replace(self, N=n, name=f"{self.name}@N{n}")


# The five workloads the library is checked and measured on.
TINY = Workload("tiny_b1h1_n128_d64", 1, 1, 128, 64, False, backward=False, seed=1000)
MEDIUM_D64 = Workload("b4h16_n1024_d64", 4, 16, 1024, 64, False, seed=1001)
CAUSAL_OUTLIERS = Workload("b2h32_n4096_d128_causal_outliers", 2, 32, 4096, 128, True,
                           outlier_frac=0.01, outlier_mult=20.0, seed=1002)
SWEEP_D128 = Workload("b8h16_n2048_d128_half", 8, 16, 2048, 128, False, value_scale=0.5,
                      backward=False, seed=1003)
SWEEP_NS = (512, 1024, 2048)
LONG_CAUSAL = Workload("b1h16_n16384_d128_causal", 1, 16, 16384, 128, True, seed=1004,
                       check_rows=256)

ALL = (TINY, MEDIUM_D64, CAUSAL_OUTLIERS, SWEEP_D128, LONG_CAUSAL)
BY_NAME = {w.name: w for w in ALL}


def make_inputs(w: Workload, seed: int | None = None, with_grad: bool | None = None):
    """Return dict(q, k, v[, do]) of contiguous bf16 CPU tensors [B,H,N,d]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    shape = (w.B, w.H, w.N, w.d)
    names = ["q", "k", "v"]
    if w.backward if with_grad is None else with_grad:
        names.append("do")
    t = {n: torch.randn(shape, generator=g, dtype=torch.float32) * w.value_scale
         for n in names}
    if w.outlier_frac > 0:
        n_out = int(round(w.outlier_frac * w.N))
        for name in ("q", "k"):
            for b in range(w.B):
                for h in range(w.H):
                    rows = torch.randperm(w.N, generator=g)[:n_out]
                    t[name][b, h, rows] *= w.outlier_mult
    if w.entry_outlier_frac > 0:
        for name in ("q", "k", "v"):
            u = torch.rand(shape, generator=g, dtype=torch.float32)
            z = torch.randn(shape, generator=g, dtype=torch.float32) * w.entry_outlier_std
            t[name] = torch.where(u < w.entry_outlier_frac, z, t[name])
    return {n: x.to(torch.bfloat16).contiguous() for n, x in t.items()}


def make_inputs_device(w: Workload, device, seed: int | None = None,
                       with_grad: bool | None = None):
    """Return dict(q, k, v[, do]) of contiguous bf16 tensors [B,H,N,d] on ``device``."""
    if w.outlier_frac > 0 or w.entry_outlier_frac > 0:
        raise ValueError("make_inputs_device draws no outliers")
    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)
    shape = (w.B, w.H, w.N, w.d)
    names = ["q", "k", "v"]
    if w.backward if with_grad is None else with_grad:
        names.append("do")
    out = {}
    for n in names:
        x = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
        x.mul_(w.value_scale)
        out[n] = x.to(torch.bfloat16).contiguous()
        del x
    return out


def random_signs(d: int, seed: int) -> torch.Tensor:
    """fp32 [d] of +-1, each sign an independent fair draw (CPU tensor)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    bits = torch.randint(0, 2, (d,), generator=g)
    return (bits * 2 - 1).to(torch.float32)


def sample_rows(w: Workload, count: int, seed: int, causal_spread: bool = True):
    """Seeded row indices [B, H, count] for row-subset checks.

    The first and last rows are always included (edges of the mask and of a
    partial last tile); the rest are drawn uniformly without replacement.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    out = torch.empty((w.B, w.H, count), dtype=torch.long)
    for b in range(w.B):
        for h in range(w.H):
            r = torch.randperm(w.N, generator=g)[:count]
            if causal_spread and count >= 2:
                r[0], r[1] = 0, w.N - 1
                r = torch.unique(r)
                while r.numel() < count:
                    extra = torch.randint(0, w.N, (count - r.numel(),), generator=g)
                    r = torch.unique(torch.cat([r, extra]))
            out[b, h] = torch.sort(r[:count]).values
    return out
