"""Seeded synthetic inputs for the SANATAN p=1 attention workloads.

This module only draws random numbers and fixes shapes; it holds none of the
method's arithmetic, so both the CUDA path and the float64 oracle can consume
its tensors without sharing any computation.

Recipe (one torch ``Generator`` per workload, seed = 1000 + workload index,
values drawn in float32 and then cast to the workload's input dtype):
  * omega ~ U(-pi, pi) of shape [H, d] (drawn first),
  * q, k ~ N(0, 1) of shape [B, H, T, d], v ~ N(0, 1) of shape [B, H, T, dv],
    then dO ~ N(0, 1) for the training workload,
  * gamma = 4 for every head,
  * phi (the per-dimension rotation rate) is either 0 or 10000^(-a/d) for
    a = 0..d-1, computed in float64 and rounded once to float32, identical for
    every head.

The shapes stand in for the 184M-parameter model of the SANATAN paper
(12 layers x 12 heads, d = 64); no dataset or trained weight is involved.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    B: int
    H: int
    T: int
    d: int = 64
    dv: int = 64
    dtype: str = "bf16"          # input dtype of q, k, v: "f32" or "bf16"
    phi_kind: str = "geometric"  # "zero" or "geometric" (10000^(-a/d))
    gamma0: float = 4.0
    extra: dict = field(default_factory=dict)

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def token_heads(self) -> int:
        return self.B * self.H * self.T


# The five workloads.  Index 0 is the small exact-arithmetic case, 1 the layer
# forward at the 184M model's shape, 2 the long prefill, 3 the batched decode
# (12 layers x 12 heads = 144 independent state slots per sequence, prefilled
# with 4096 tokens and then stepped 1024 times), 4 the training step.
TINY = Workload("tiny_f32_T256", 0, B=1, H=1, T=256, dtype="f32", phi_kind="zero")
LAYER = Workload("layer_fwd_B4_H12_T2048", 1, B=4, H=12, T=2048)
LONG = Workload("long_prefill_B1_H12_T32768", 2, B=1, H=12, T=32768)
DECODE = Workload("decode_L12xH12", 3, B=1, H=144, T=4096,
                  extra=dict(steps=1024, batches=(1, 64), layers=12, heads=12))
TRAIN = Workload("train_fwd_bwd_B8_H12_T4096", 4, B=8, H=12, T=4096)

ALL = (TINY, LAYER, LONG, DECODE, TRAIN)

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def shard_seed(seed: int, shard: int) -> int:
    """Seed of the data of replica ``shard`` (shard 0 keeps the workload's)."""
    return int(seed) + 1_000_003 * int(shard)


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def rates(H: int, d: int, kind: str) -> torch.Tensor:
    """Rotation rates phi [H, d] as float32."""
    if kind == "zero":
        return torch.zeros(H, d, dtype=torch.float32)
    if kind == "geometric":
        row = torch.tensor([10000.0 ** (-a / d) for a in range(d)], dtype=torch.float64)
        return row.to(torch.float32).unsqueeze(0).repeat(H, 1).contiguous()
    raise ValueError(kind)


def params(H: int, d: int, phi_kind: str, gen: torch.Generator, gamma0: float = 4.0,
           device="cpu"):
    """gamma [H], omega [H, d], phi [H, d]; all float32 on ``device``."""
    omega = (torch.rand(H, d, generator=gen, dtype=torch.float32, device=gen.device)
             * (2.0 * math.pi) - math.pi)
    gamma = torch.full((H,), float(gamma0), dtype=torch.float32)
    phi = rates(H, d, phi_kind)
    return gamma.to(device), omega.to(device), phi.to(device)


def normal(shape, gen: torch.Generator, dtype: str, device=None) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32, device=gen.device)
    x = x.to(TORCH_DTYPE[dtype])
    return x if device is None else x.to(device)


def make(w: Workload, device="cpu", B=None, H=None, T=None, with_grad_out=False, shard=0):
    """Inputs of workload ``w`` (optionally with B/H/T overridden for a
    reduced-size case that keeps the same distributions).  Random numbers are
    drawn on ``device`` (a CUDA generator for device tensors, so that large
    cases need no host copy); the returned dict holds q, k, v (and dO), gamma,
    omega, phi, and the sizes.  ``shard`` > 0 draws another batch of q, k, v
    (a data-parallel replica's own sequences) with the same gamma, omega, phi."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    T = w.T if T is None else T
    gen = generator(w.seed, device)
    gamma, omega, phi = params(H, w.d, w.phi_kind, gen, w.gamma0, device)
    if shard:
        gen = generator(shard_seed(w.seed, shard), device)
    out = dict(B=B, H=H, T=T, d=w.d, dv=w.dv, dtype=w.dtype,
               gamma=gamma, omega=omega, phi=phi)
    out["q"] = normal((B, H, T, w.d), gen, w.dtype)
    out["k"] = normal((B, H, T, w.d), gen, w.dtype)
    out["v"] = normal((B, H, T, w.dv), gen, w.dtype)
    if with_grad_out:
        out["dO"] = normal((B, H, T, w.dv), gen, w.dtype)
    return out


def decode_tokens(n_slots: int, d: int, dv: int, steps: int, gen: torch.Generator):
    """Fresh float32 N(0,1) q, k [steps, n_slots, d] and v [steps, n_slots, dv]
    for the decode steps that follow a prefill."""
    q = torch.randn(steps, n_slots, d, generator=gen, dtype=torch.float32, device=gen.device)
    k = torch.randn(steps, n_slots, d, generator=gen, dtype=torch.float32, device=gen.device)
    v = torch.randn(steps, n_slots, dv, generator=gen, dtype=torch.float32, device=gen.device)
    return q, k, v


def to_f64(x: torch.Tensor):
    """Exact float64 numpy copy (bf16 and f32 values promote exactly)."""
    return x.detach().to("cpu", torch.float64).numpy()
