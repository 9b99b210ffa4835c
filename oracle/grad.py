"""Gradient oracle of the causal ZeroS layer: plain fp64 PyTorch on the CPU.

TEST INFRASTRUCTURE ONLY.  Only the tests use this module; it shares no code with the CUDA
path (nor with the C++ oracle, against which its forward is checked).

The forward below is the definition written out, O(N^2 d) (Paper-Notes "ZeroS: Zero-Sum Linear
Attention for Efficient Transformers", method details):
  * deviation logits: s_i = -(1/sqrt d) u_i ubar_i^T, ubar_i = (e^tau mu + sum_{j<=i} u_j) /
    (e^tau + i) ("deviation logits");
  * zero-sum weights: softmax_{t,i} = e^{s_i}/E_t, delta_{t,i} = s_i - P_t/t,
    eps_{t,i} = softmax_{t,i} - 1/t - delta_{t,i}/t, w_{t,i} = sig1_t delta_{t,i}/t +
    sigh_t eps_{t,i} (+ sig0_t/t with the optional zero-order gate) ("zero-order removal");
  * angular factor: cos theta_{t,i} = q_hat_t R_{t-i} k_hat_i^T, applied as absolute rotations
    of the unit vectors ("radial-angular decoupling", RoPE form);
  * o_t = sum_{i<=t} w_{t,i} cos theta_{t,i} v_i.
The readings are those of the C++ oracle (half-split rotary pairs, theta_a = base^{-2a/d},
token t at position t - 1, x_hat = x / ||x||).  The gradients are torch.autograd's derivatives
of this fp64 forward; tests pin them against central finite differences.
"""
from __future__ import annotations

import math

import numpy as np
import torch


def _t(x):
    if isinstance(x, torch.Tensor):
        return x.detach().cpu().double().clone()
    return torch.as_tensor(np.asarray(x), dtype=torch.float64).clone()


def _rotate(x, base):
    """Rotary map of rows x[..., n, d] at positions n = 0 .. N-1 (half-split pairs)."""
    N, d = x.shape[-2], x.shape[-1]
    half = d // 2
    theta = base ** (-2.0 * torch.arange(half, dtype=torch.float64) / d)
    ang = torch.arange(N, dtype=torch.float64)[:, None] * theta[None, :]
    c, s = torch.cos(ang), torch.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return torch.cat([a * c - b * s, a * s + b * c], dim=-1)


def forward(q, k, v, u, g1, gh, mu, tau, *, rope=False, rope_base=10000.0, g0=None):
    """Causal forward of the definition, fp64 torch tensors in, [B,H,N,d] out (differentiable)."""
    B, H, N, d = q.shape
    et = torch.exp(tau)[None, :, None, None]                         # [1,H,1,1]
    idx = torch.arange(1, N + 1, dtype=torch.float64)                # t (1-based)
    ubar = (et * mu[None, :, None, :] + torch.cumsum(u, dim=2)) / (et + idx[:, None])
    s = -(u * ubar).sum(-1) / math.sqrt(d)                          # [B,H,N]
    mask = torch.tril(torch.ones(N, N, dtype=torch.bool))            # i <= t
    es = torch.exp(s)
    E = torch.cumsum(es, dim=2)
    P = torch.cumsum(s, dim=2)
    tt = idx[None, None, :, None]                                    # t as [.., t, 1]
    soft = es[:, :, None, :] / E[..., None]
    delta = s[:, :, None, :] - P[..., None] / tt
    eps = soft - 1.0 / tt - delta / tt
    sig1 = torch.sigmoid(g1)[..., None]
    sigh = torch.sigmoid(gh)[..., None]
    w = sig1 * delta / tt + sigh * eps
    if g0 is not None:
        w = w + torch.sigmoid(g0)[..., None] / tt
    w = torch.where(mask, w, torch.zeros((), dtype=torch.float64))
    qn = q / q.norm(dim=-1, keepdim=True)
    kn = k / k.norm(dim=-1, keepdim=True)
    if rope:
        qn, kn = _rotate(qn, rope_base), _rotate(kn, rope_base)
    cos = qn @ kn.transpose(-1, -2)                                   # [B,H,N,N]
    return (w * cos) @ v


def backward(q, k, v, u, g1, gh, mu, tau, do, *, rope=False, rope_base=10000.0, g0=None):
    """Gradients of sum(o * do) with respect to every input: a dict of fp64 numpy arrays with
    keys q, k, v, u, g1, gh, mu, tau (and g0 when given)."""
    names = ["q", "k", "v", "u", "g1", "gh", "mu", "tau"]
    xs = [_t(x).requires_grad_(True) for x in (q, k, v, u, g1, gh, mu, tau)]
    g0t = None
    if g0 is not None:
        g0t = _t(g0).requires_grad_(True)
        names.append("g0")
        xs.append(g0t)
    o = forward(*xs[:8], rope=rope, rope_base=rope_base, g0=g0t)
    grads = torch.autograd.grad(o, xs, grad_outputs=_t(do))
    return {n: g.numpy() for n, g in zip(names, grads)}
