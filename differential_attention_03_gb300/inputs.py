"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module only draws random numbers and casts them; it holds none of the
method's arithmetic (no lambda, no softmax, no norm) and imports nothing else
from this package, so that the CUDA path and the CPU oracle can both be fed
from it without sharing any computation.

Recipe (one torch generator per call, seeded with the workload's seed; draws
in the order listed, each an fp32 tensor then cast to the workload's dtype):
  V1:  Q1, Q2, K1, K2 ~ N(0,1) [B, n, H, d]; V ~ N(0,1) [B, n, H, 2d];
       lq1, lk1, lq2, lk2 ~ N(0, 0.1^2) [d] (fp32);
       gamma = 1, or ~ U(0.9, 1.1) [2d] (fp32).
  V2:  Q ~ N(0,1) [B, n, Hq, d]; K, V ~ N(0,1) [B, n, Hkv, d];
       lambda logits ~ N(0,1) [Hq/2] (fp32), one per head pair.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, dtype, causal flag, layer index, seed."""

    name: str
    kind: str  # "v1" or "v2"
    dtype: str  # "f32" or "bf16"
    B: int
    n: int
    d: int
    H: int = 0  # V1 diff heads
    Hq: int = 0  # V2 query heads
    Hkv: int = 0  # V2 KV heads
    layer: int = 1  # V1 layer index l (1-based)
    gamma: str = "ones"  # "ones" or "uniform"
    causal: bool = True
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


# The five workloads the measurements are quoted on (seed = workload number).
WORKLOADS = {
    1: Workload("v1-f32-B1H1-n128-d64", "v1", "f32", B=1, n=128, d=64, H=1, layer=4, seed=1),
    2: Workload("v1-bf16-B4H16-n2048-d64", "v1", "bf16", B=4, n=2048, d=64, H=16, layer=1, seed=2),
    3: Workload("v1-bf16-B2H12-n4096-d128", "v1", "bf16", B=2, n=4096, d=128, H=12, layer=12,
                gamma="uniform", seed=3),
    4: Workload("v1-bf16-B1H12-n65536-d128", "v1", "bf16", B=1, n=65536, d=128, H=12, layer=20, seed=4),
    5: Workload("v2-bf16-B8Hq32Hkv16-n8192-d128", "v2", "bf16", B=8, n=8192, d=128, Hq=32, Hkv=16, seed=5),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_v1(w: Workload, device="cpu") -> dict:
    """Draw the V1 tensors of workload ``w`` on ``device`` (see module docstring)."""
    g = _gen(w.seed, device)
    dt = w.torch_dtype

    def randn(*shape, std=1.0, cast=True):
        x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            x = x * std
        return x.to(dt) if cast else x

    shp = (w.B, w.n, w.H, w.d)
    out = {
        "q1": randn(*shp), "q2": randn(*shp), "k1": randn(*shp), "k2": randn(*shp),
        "v": randn(w.B, w.n, w.H, 2 * w.d),
    }
    for name in ("lq1", "lk1", "lq2", "lk2"):
        out[name] = randn(w.d, std=0.1, cast=False)
    if w.gamma == "uniform":
        u = torch.rand(2 * w.d, generator=g, device=device, dtype=torch.float32)
        out["gamma"] = 0.9 + 0.2 * u
    else:
        out["gamma"] = torch.ones(2 * w.d, device=device, dtype=torch.float32)
    return out


def make_v2(w: Workload, device="cpu") -> dict:
    """Draw the V2 tensors of workload ``w`` on ``device`` (see module docstring)."""
    g = _gen(w.seed, device)
    dt = w.torch_dtype

    def randn(*shape, cast=True):
        x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
        return x.to(dt) if cast else x

    return {
        "q": randn(w.B, w.n, w.Hq, w.d),
        "k": randn(w.B, w.n, w.Hkv, w.d),
        "v": randn(w.B, w.n, w.Hkv, w.d),
        "lam_logits": randn(w.Hq // 2, cast=False),
    }


def shrink(w: Workload, **changes) -> Workload:
    """A copy of ``w`` with some fields replaced (smaller parity cases)."""
    d = dict(w.__dict__)
    d.update(changes)
    return Workload(**d)
