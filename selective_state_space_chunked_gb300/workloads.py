"""Seeded synthetic inputs for the three scans.

This module only draws random numbers and applies the input preparation that
sits OUTSIDE the scans (sigmoid-activated gates, the lower-bounded HGRN2 gate,
the multi-scale A_log parameter).  It holds none of the recurrences: both the
CUDA library and the float64 oracle receive what it returns.

Distributions follow the source pages' layer definitions:

* RG-LRU (lrnnx ``RGLRU.__init__`` / ``forward``): x, r_pre, i_pre ~ N(0,1);
  r = sigmoid(r_pre), i = sigmoid(i_pre) (the recurrent and input gates);
  per-channel base a ~ U(0.9, 0.999), ``a_log = log a``; c = 8.
* Selective SSM (cortexnet ``MultiScaleSSM.__init__``): ``A_log[d, n] =
  log((n+1) * 2**s)`` for channel d in scale s (d_inner split evenly over the
  scales); D skip = 1; the pre-softplus step ``dt_pre = u + e`` where
  u ~ U(ln 1e-3, ln 1e-1) is the dt bias initialisation range and
  e ~ N(0, variance 0.1) stands in for ``dt_proj(x)``; x, z, B_t, C_t ~ N(0,1).
* HGRN2 (HGRN2 Attention page): q, k, v ~ N(0, variance 1/128); forget
  pre-activation f ~ N(2, 1); ``g = lb + (1 - lb) * sigmoid(f)``, lb = 0.2.

Every tensor is drawn from one ``torch.Generator`` seeded with the config's
seed, in the fixed order written in each function.  Generation runs on the
requested device (CPU for oracle-sized cases; the GPU generator for the
full-size benchmark, whose oracle samples are then copied back to the host).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import torch

__all__ = [
    "WORKLOADS", "Config", "multiscale_A_log", "rglru_inputs",
    "selective_inputs", "hgrn2_inputs", "make_inputs",
]


@dataclass(frozen=True)
class Config:
    """One workload: which scan, its sizes, I/O dtype and seed."""
    index: int
    form: str            # "rglru" | "selective" | "hgrn2"
    B: int
    L: int
    D: int               # channels (rglru/selective) or hidden size (hgrn2)
    io: str              # "f32" | "bf16"
    seed: int
    N: int = 16          # selective state size
    n_scales: int = 4    # selective multi-scale A
    H: int = 16          # hgrn2 heads
    head_dim: int = 128  # hgrn2 head dim (dk = dv)
    chunk: int = 64      # hgrn2 chunk length on the GPU path
    lb: float = 0.2      # hgrn2 gate lower bound
    with_h0: bool = False

    @property
    def name(self) -> str:
        if self.form == "hgrn2":
            return (f"hgrn2_{self.io}_B{self.B}_L{self.L}_H{self.H}"
                    f"_d{self.head_dim}")
        extra = f"_N{self.N}" if self.form == "selective" else ""
        return f"{self.form}_{self.io}_B{self.B}_L{self.L}_D{self.D}{extra}"

    @property
    def token_channels(self) -> int:
        """Token-channel steps one pass processes (B * L * channels)."""
        return self.B * self.L * self.D


# The five workloads the pages' layers are sized for, by name (the index is
# the seed).
WORKLOADS = {
    "rglru_f32_small": Config(0, "rglru", B=2, L=128, D=64, io="f32", seed=0),
    "selective_f32": Config(1, "selective", B=2, L=1024, D=1536, io="f32", seed=1),
    "rglru_bf16": Config(2, "rglru", B=8, L=4096, D=2560, io="bf16", seed=2, with_h0=True),
    "selective_bf16": Config(3, "selective", B=4, L=16384, D=4096, io="bf16", seed=3,
                             with_h0=True),
    "hgrn2_bf16": Config(4, "hgrn2", B=4, L=4096, D=2048, io="bf16", seed=4, H=16,
                         head_dim=128),
}


def _dtype(io: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[io]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def multiscale_A_log(D: int, N: int, n_scales: int = 4) -> torch.Tensor:
    """The multi-scale parameter of cortexnet ``MultiScaleSSM.__init__``.

    d_inner = D channels are split into ``n_scales`` equal groups; group s
    holds ``A[d, n] = (n + 1) * 2**s`` and the stored parameter is
    ``log(A)`` in float32, shape (D, N).
    """
    if D % n_scales:
        raise ValueError("D must be divisible by n_scales")
    per = D // n_scales
    parts = []
    for s in range(n_scales):
        base = torch.arange(1, N + 1, dtype=torch.float32) * (2.0 ** s)
        parts.append(base.unsqueeze(0).expand(per, N))
    return torch.log(torch.cat(parts, dim=0)).contiguous()


def rglru_inputs(B: int, L: int, D: int, seed: int, io: str = "f32",
                 with_h0: bool = False, device="cpu", c: float = 8.0) -> dict:
    """RG-LRU inputs.  Draw order: x, r_pre, i_pre (each (B, L, D)), a (D),
    then h0 (B, D) when requested."""
    g = _gen(seed, device)
    x = torch.randn(B, L, D, generator=g, device=device)
    r_pre = torch.randn(B, L, D, generator=g, device=device)
    i_pre = torch.randn(B, L, D, generator=g, device=device)
    a = 0.9 + (0.999 - 0.9) * torch.rand(D, generator=g, device=device)
    h0 = torch.randn(B, D, generator=g, device=device) if with_h0 else None
    dt = _dtype(io)
    return {
        "x": x.to(dt).contiguous(),
        "r": torch.sigmoid(r_pre).to(dt).contiguous(),
        "i": torch.sigmoid(i_pre).to(dt).contiguous(),
        "a_log": torch.log(a).float().contiguous(),
        "c": float(c),
        "h0": h0,
    }


def selective_inputs(B: int, L: int, D: int, seed: int, io: str = "f32",
                     N: int = 16, n_scales: int = 4, with_h0: bool = False,
                     device="cpu") -> dict:
    """Selective-SSM inputs.  Draw order: x, z (B, L, D); Bm, Cm (B, L, N);
    u (B, L, D) uniform; e (B, L, D) normal; then h0 (B, D, N) when
    requested.  ``dt`` is the pre-softplus step; call with
    ``dt_softplus=True``."""
    g = _gen(seed, device)
    x = torch.randn(B, L, D, generator=g, device=device)
    z = torch.randn(B, L, D, generator=g, device=device)
    Bm = torch.randn(B, L, N, generator=g, device=device)
    Cm = torch.randn(B, L, N, generator=g, device=device)
    lo, hi = math.log(1e-3), math.log(1e-1)
    u = lo + (hi - lo) * torch.rand(B, L, D, generator=g, device=device)
    e = math.sqrt(0.1) * torch.randn(B, L, D, generator=g, device=device)
    dt_pre = u.add_(e)
    del e
    h0 = torch.randn(B, D, N, generator=g, device=device) if with_h0 else None
    dt = _dtype(io)
    return {
        "x": x.to(dt).contiguous(),
        "dt": dt_pre.to(dt).contiguous(),
        "z": z.to(dt).contiguous(),
        "Bm": Bm.to(dt).contiguous(),
        "Cm": Cm.to(dt).contiguous(),
        "A_log": multiscale_A_log(D, N, n_scales).to(device),
        "Dskip": torch.ones(D, device=device),
        "h0": h0,
        "dt_softplus": True,
    }


def hgrn2_inputs(B: int, L: int, H: int, head_dim: int, seed: int,
                 io: str = "bf16", lb: float = 0.2, with_S0: bool = False,
                 device="cpu") -> dict:
    """HGRN2 inputs.  Draw order: q, k, v (B, L, H*head_dim), f (same), then
    S0 (B, H, head_dim, head_dim) when requested."""
    g = _gen(seed, device)
    hid = H * head_dim
    std = math.sqrt(1.0 / 128.0)
    q = std * torch.randn(B, L, hid, generator=g, device=device)
    k = std * torch.randn(B, L, hid, generator=g, device=device)
    v = std * torch.randn(B, L, hid, generator=g, device=device)
    f = 2.0 + torch.randn(B, L, hid, generator=g, device=device)
    S0 = (torch.randn(B, H, head_dim, head_dim, generator=g, device=device)
          if with_S0 else None)
    gate = lb + (1.0 - lb) * torch.sigmoid(f)
    dt = _dtype(io)
    return {
        "q": q.to(dt).contiguous(),
        "k": k.to(dt).contiguous(),
        "v": v.to(dt).contiguous(),
        "g": gate.to(dt).contiguous(),
        "S0": S0,
        "H": H,
    }


def make_inputs(cfg: Config, device="cpu", B: Optional[int] = None,
                L: Optional[int] = None) -> dict:
    """Inputs of a workload, optionally with B or L overridden (same seed and
    distributions; used for oracle-sized parity cases)."""
    B = cfg.B if B is None else B
    L = cfg.L if L is None else L
    if cfg.form == "rglru":
        return rglru_inputs(B, L, cfg.D, cfg.seed, cfg.io, cfg.with_h0, device)
    if cfg.form == "selective":
        return selective_inputs(B, L, cfg.D, cfg.seed, cfg.io, cfg.N,
                                cfg.n_scales, cfg.with_h0, device)
    if cfg.form == "hgrn2":
        return hgrn2_inputs(B, L, cfg.H, cfg.head_dim, cfg.seed, cfg.io,
                            cfg.lb, device=device)
    raise ValueError(cfg.form)
