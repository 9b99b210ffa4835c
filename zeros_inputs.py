"""Seeded synthetic inputs for the ZeroS hot path.

This module holds no part of the method's arithmetic: it only draws random tensors with the
shapes and distributions of the workloads below and casts them to the storage dtype.  Both
the oracle side and the CUDA side of every test consume exactly the tensors produced here.

Recipe:
  * q, k, v, u ~ N(0, 1) drawn in fp32 with a torch.Generator seeded per workload, then
    rounded to the storage dtype (bf16 round-to-nearest-even, or kept fp32).
  * g1, gh (gate logits) ~ N(0, gate_var) in fp32.
  * mu ~ N(0, 1) per head ([H, d] fp32); tau ~ U(-1, 1) per head ([H] fp32) unless fixed.
  * Long-context workload: every token's u row is multiplied by one c ~ U(0.5, 2) before
    rounding, to widen the spread of the deviation logits.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str = "bf16"        # storage dtype of q, k, v, u and out: "bf16" or "f32"
    causal: bool = True
    rope: bool = False
    rope_base: float = 10000.0
    gate_var: float = 1.0
    tau: float | None = None   # fixed tau for every head, or None for U(-1, 1)
    u_scale: tuple | None = None  # per-token U(lo, hi) multiplier of u
    seed: int = 0
    decode_steps: int = 0      # recurrent-decode workloads: tokens decoded after the prefill

    def tokens(self) -> int:
        return self.B * self.N

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads of the benchmark specification, by what they are.
CAUSAL_F32_SMALL = Workload("causal-f32 B1 H1 N256 d32", 1, 1, 256, 32, dtype="f32",
                            tau=0.0, seed=0)
CAUSAL_ROPE_B8H8N4096D64 = Workload("causal-rope bf16 B8 H8 N4096 d64", 8, 8, 4096, 64,
                                    rope=True, seed=2)
ENCODER_VIT_B256H3N197D64 = Workload("encoder bf16 B256 H3 N197 d64", 256, 3, 197, 64,
                                     causal=False, seed=3)
LONG_ROPE_B2H16N65536D128 = Workload("causal-rope bf16 B2 H16 N65536 d128", 2, 16, 65536, 128,
                                     rope=True, gate_var=2.0, u_scale=(0.5, 2.0), seed=4)
DECODE_B256H32D128 = Workload("decode bf16 B256 H32 d128 prefill 8192 + 1024 steps", 256, 32,
                              8192, 128, seed=5, decode_steps=1024)

ALL = [CAUSAL_F32_SMALL, CAUSAL_ROPE_B8H8N4096D64, ENCODER_VIT_B256H3N197D64,
       LONG_ROPE_B2H16N65536D128, DECODE_B256H32D128]


def storage_dtype(w: Workload) -> torch.dtype:
    return torch.bfloat16 if w.dtype == "bf16" else torch.float32


def make(w: Workload, device="cpu", N: int | None = None, B: int | None = None) -> dict:
    """Draw one set of inputs for workload ``w``.

    ``N`` / ``B`` override the sequence length / batch (e.g. prefill plus decode tokens).
    Tensors are contiguous and live on ``device``; the generator runs on that device, so the
    values depend on the device (each test uses one device as its source of truth)."""
    B = w.B if B is None else B
    N = w.N if N is None else N
    H, d = w.H, w.d
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    sd = storage_dtype(w)

    def normal(shape, std=1.0):
        return torch.randn(shape, generator=g, device=dev, dtype=torch.float32) * std

    q = normal((B, H, N, d)).to(sd)
    k = normal((B, H, N, d)).to(sd)
    v = normal((B, H, N, d)).to(sd)
    u = normal((B, H, N, d))
    if w.u_scale is not None:
        lo, hi = w.u_scale
        c = torch.rand((B, H, N, 1), generator=g, device=dev, dtype=torch.float32)
        u = u * (lo + (hi - lo) * c)
    u = u.to(sd)
    g1 = normal((B, H, N), std=w.gate_var ** 0.5)
    gh = normal((B, H, N), std=w.gate_var ** 0.5)
    mu = normal((H, d))
    if w.tau is None:
        tau = torch.rand((H,), generator=g, device=dev, dtype=torch.float32) * 2.0 - 1.0
    else:
        tau = torch.full((H,), float(w.tau), device=dev, dtype=torch.float32)
    return dict(q=q, k=k, v=v, u=u, g1=g1, gh=gh, mu=mu, tau=tau)


def decode_tokens(w: Workload, step: int, device="cpu") -> dict:
    """Inputs for one recurrent-decode step: q,k,v,u [B,H,d], g1,gh [B,H] (seeded per step)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed * 1_000_003 + 7919 * (step + 1))
    sd = storage_dtype(w)
    B, H, d = w.B, w.H, w.d

    def normal(shape, std=1.0):
        return torch.randn(shape, generator=g, device=dev, dtype=torch.float32) * std

    out = {n: normal((B, H, d)).to(sd) for n in ("q", "k", "v", "u")}
    out["g1"] = normal((B, H), std=w.gate_var ** 0.5)
    out["gh"] = normal((B, H), std=w.gate_var ** 0.5)
    return out


def sample_heads(w: Workload, count: int, seed: int = 12345) -> list:
    """A seeded subset of (b, h) pairs used where the oracle cannot run every sequence."""
    g = torch.Generator()
    g.manual_seed(seed + w.seed)
    total = w.B * w.H
    idx = torch.randperm(total, generator=g)[: min(count, total)].tolist()
    return sorted((i // w.H, i % w.H) for i in idx)
