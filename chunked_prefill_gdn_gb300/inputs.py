"""Seeded synthetic inputs for the GDN chunked-prefill workloads.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle take their inputs
from here.

Shapes follow the FLA convention that the FlashQLA talk ("Qwen系列模型线性注意力
高性能优化实践", API paragraph) says the library keeps: q, k are [B, T, H, dk],
v is [B, T, H, dv], the log-gate g and the update gate beta are [B, T, H]
(fp32), a varlen batch is packed with B = 1 plus int32 cu_seqlens [N + 1], and
the state is [N, H, dk, dv] (fp32).

Recipes (all draws are standard normal unless stated; the order of draws is
fixed: lengths (varlen only), q, k, v, beta logits, gate noise, per-head a_h,
initial state):
  q, k   ~ N(0, 1), L2-normalised over dk in fp32, then cast to the input dtype
  v      ~ N(0, 1), cast to the input dtype
  beta   = sigmoid(N(0, 1))                                (fp32)
  g      = -exp(a_h) * softplus(N(0, 1)),  a_h ~ U(lo, hi) per head   (fp32)
           ("tiny" uses g = -0.1 * softplus(N(0, 1)));
           heads listed in zero_gate_heads get g == 0 exactly (alpha == 1)
  S0     ~ N(0, s0_std^2) fp32, or None (zero state)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional, Sequence

import torch

__all__ = ["WorkloadConfig", "CONFIGS", "config", "make_inputs", "make_grad_inputs", "varlen_lengths"]


@dataclass(frozen=True)
class WorkloadConfig:
    name: str
    B: int
    T: int                      # per-sequence length (batched) or total tokens (varlen)
    H: int
    dk: int
    dv: int
    dtype: str                  # "bf16" or "f32" for q/k/v/o
    seed: int
    gate: str = "decay"         # "decay" or "tiny"
    a_range: tuple = (-4.0, -1.0)
    zero_gate_heads: tuple = ()
    s0_std: Optional[float] = None
    n_seqs: Optional[int] = None  # varlen when set (B must be 1)
    len_mu: float = 8.0
    len_sigma: float = 1.0
    len_min: int = 64
    len_max: int = 32768
    C: int = 64

    @property
    def varlen(self) -> bool:
        return self.n_seqs is not None

    @property
    def total_tokens(self) -> int:
        return self.T if self.varlen else self.B * self.T

    @property
    def num_seqs(self) -> int:
        return self.n_seqs if self.varlen else self.B

    def scaled(self, **kw) -> "WorkloadConfig":
        """A copy with some fields replaced (reduced sizes for parity cases)."""
        return replace(self, **kw)


# The five synthetic workloads. Index 1 is the headline layer shape.
CONFIGS = {
    0: WorkloadConfig("tiny", B=1, T=256, H=2, dk=32, dv=32, dtype="f32", seed=0, gate="tiny"),
    1: WorkloadConfig("layer", B=4, T=8192, H=32, dk=128, dv=128, dtype="bf16", seed=1,
                      a_range=(-4.0, -1.0)),
    2: WorkloadConfig("long", B=1, T=131072, H=8, dk=128, dv=128, dtype="bf16", seed=2,
                      a_range=(-4.0, -1.0), zero_gate_heads=(0, 1, 2), s0_std=0.02),
    3: WorkloadConfig("varlen", B=1, T=262144, H=16, dk=128, dv=128, dtype="bf16", seed=3,
                      a_range=(-4.0, -1.0), n_seqs=64),
    4: WorkloadConfig("1m_mix", B=1, T=1048576, H=16, dk=128, dv=128, dtype="bf16", seed=4,
                      a_range=(-3.0, -1.0), zero_gate_heads=(0, 1, 2, 3, 4), s0_std=0.02),
}


def config(idx: int) -> WorkloadConfig:
    return CONFIGS[idx]


def _torch_dtype(name: str):
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def varlen_lengths(n: int, total: int, seed: int, mu: float = 8.0, sigma: float = 1.0,
                   lo: int = 64, hi: int = 32768) -> list:
    """Sequence lengths ~ lognormal(mu, sigma), clipped to [lo, hi], rescaled so
    that they sum to `total` exactly.  The remainder after flooring goes +1 to the
    longest sequences that still have room (or -1 from the longest above lo)."""
    if n * lo > total or n * hi < total:
        raise ValueError("cannot pack %d sequences of length [%d, %d] into %d" % (n, lo, hi, total))
    gen = torch.Generator().manual_seed(seed)
    raw = torch.exp(mu + sigma * torch.randn(n, generator=gen, dtype=torch.float64))
    raw = raw.clamp(lo, hi)
    lens = (raw * (total / raw.sum())).floor().clamp(lo, hi).to(torch.int64).tolist()
    order = sorted(range(n), key=lambda i: (-lens[i], i))
    diff = total - sum(lens)
    while diff != 0:
        moved = False
        for i in order:
            if diff > 0 and lens[i] < hi:
                lens[i] += 1
                diff -= 1
                moved = True
            elif diff < 0 and lens[i] > lo:
                lens[i] -= 1
                diff += 1
                moved = True
            if diff == 0:
                break
        if not moved:
            raise RuntimeError("length fix-up did not converge")
    return lens


def _normal(shape, gen, device):
    return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)


def make_inputs(cfg: WorkloadConfig, device="cpu", chunk_tokens: int = 1 << 18) -> dict:
    """Draw one workload.  Returns a dict with
    q, k [B,T,H,dk]; v [B,T,H,dv] (cfg.dtype); g, beta [B,T,H] fp32;
    initial_state [N,H,dk,dv] fp32 or None; cu_seqlens int32 [N+1] or None;
    scale (float, dk^-0.5) and the config.

    Large tensors are drawn `chunk_tokens` tokens at a time so the fp32
    temporaries stay small.  The values are a deterministic function of
    (config, device type, chunk_tokens); CPU and CUDA generators give different
    streams, so a test that compares two paths hands both the same tensors.
    """
    device = torch.device(device)
    gen = torch.Generator(device=device).manual_seed(cfg.seed)
    dt = _torch_dtype(cfg.dtype)
    B, H, dk, dv = cfg.B, cfg.H, cfg.dk, cfg.dv
    if cfg.varlen:
        if B != 1:
            raise ValueError("varlen workloads pack into B = 1")
        lens = varlen_lengths(cfg.n_seqs, cfg.T, cfg.seed, cfg.len_mu, cfg.len_sigma,
                              cfg.len_min, cfg.len_max)
        cu = torch.zeros(cfg.n_seqs + 1, dtype=torch.int32)
        cu[1:] = torch.tensor(lens, dtype=torch.int64).cumsum(0).to(torch.int32)
        T = cfg.T
    else:
        cu = None
        T = cfg.T
    ntok = B * T

    def draw_rows(d, normalise):
        out = torch.empty(ntok, H, d, dtype=dt, device=device)
        for s in range(0, ntok, chunk_tokens):
            e = min(ntok, s + chunk_tokens)
            x = _normal((e - s, H, d), gen, device)
            if normalise:
                x = _unit_rows(x)
            out[s:e] = x.to(dt)
            del x
        return out.view(B, T, H, d)

    q = draw_rows(dk, True)
    k = draw_rows(dk, True)
    v = draw_rows(dv, False)
    beta = torch.sigmoid(_normal((ntok, H), gen, device)).view(B, T, H)
    noise = torch.nn.functional.softplus(_normal((ntok, H), gen, device))
    lo, hi = cfg.a_range
    a_h = lo + (hi - lo) * torch.rand(H, generator=gen, device=device, dtype=torch.float32)
    if cfg.gate == "tiny":
        g = -0.1 * noise
    else:
        g = -torch.exp(a_h)[None, :] * noise
    if cfg.zero_gate_heads:
        g[:, list(cfg.zero_gate_heads)] = 0.0
    g = g.contiguous().view(B, T, H)
    s0 = None
    if cfg.s0_std is not None:
        s0 = cfg.s0_std * _normal((cfg.num_seqs, H, dk, dv), gen, device)
    return dict(q=q, k=k, v=v, g=g, beta=beta, initial_state=s0,
                cu_seqlens=None if cu is None else cu.to(device),
                scale=dk ** -0.5, config=cfg)


def make_grad_inputs(cfg: WorkloadConfig, device="cpu", seed_offset: int = 1000, ds_std: float = 0.1) -> dict:
    """Upstream gradients for the backward pass of workload `cfg`: do like o
    ([B,T,H,dv], cfg.dtype, standard normal) and d_final_state like the final
    state ([N,H,dk,dv] fp32, normal with std ds_std), from their own seed."""
    device = torch.device(device)
    gen = torch.Generator(device=device).manual_seed(cfg.seed + seed_offset)
    B, T, H, dk, dv = cfg.B, cfg.T, cfg.H, cfg.dk, cfg.dv
    do = _normal((B, T, H, dv), gen, device).to(_torch_dtype(cfg.dtype))
    dsf = ds_std * _normal((cfg.num_seqs, H, dk, dv), gen, device)
    return dict(do=do, d_final_state=dsf)
