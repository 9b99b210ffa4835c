"""Pins of the gradient oracle (oracle/grad.py, CPU).

* Its forward (the definition, written in torch) equals the pinned C++ oracle's recurrence.
* Its gradients (torch.autograd of that fp64 forward) equal central finite differences of
  L = sum(o * do) for every input, with and without RoPE and the zero-order gate.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import grad as og
from tests.oracle_pins import rand_problem

NAMES = ["q", "k", "v", "u", "g1", "gh", "mu", "tau"]


def _inputs(seed, N=7, d=6, H=2):
    p = rand_problem(seed, B=1, H=H, N=N, d=d)
    return [p[n] for n in NAMES]


@pytest.mark.parametrize("rope", [False, True])
@pytest.mark.parametrize("zero_order", [False, True])
def test_forward_equals_cpp_oracle(rope, zero_order):
    args = _inputs(31, N=40, d=8)
    g0 = np.random.default_rng(32).standard_normal(args[4].shape) if zero_order else None
    ref = oracle.forward(*args, causal=True, rope=rope, rope_base=777.0, g0=g0)
    o = og.forward(*(torch.as_tensor(a, dtype=torch.float64) for a in args), rope=rope,
                   rope_base=777.0,
                   g0=None if g0 is None else torch.as_tensor(g0, dtype=torch.float64))
    assert np.abs(o.numpy() - ref).max() <= 1e-12 * max(np.abs(ref).max(), 1.0)


@pytest.mark.parametrize("rope", [False, True])
@pytest.mark.parametrize("zero_order", [False, True])
def test_gradients_equal_finite_differences(rope, zero_order):
    args = _inputs(33 + 2 * rope + zero_order)
    rng = np.random.default_rng(34)
    do = rng.standard_normal(args[0].shape)
    g0 = rng.standard_normal(args[4].shape) if zero_order else None
    grads = og.backward(*args, do, rope=rope, rope_base=50.0, g0=g0)

    def loss(vals):
        ts = [torch.as_tensor(a, dtype=torch.float64) for a in vals[:8]]
        g = None if vals[8] is None else torch.as_tensor(vals[8], dtype=torch.float64)
        o = og.forward(*ts, rope=rope, rope_base=50.0, g0=g)
        return float((o.numpy() * do).sum())

    vals = list(args) + [g0]
    names = NAMES + (["g0"] if zero_order else [])
    h = 1e-5
    for n in names:
        pos = names.index(n)
        x = vals[pos]
        flat_idx = rng.choice(x.size, size=min(5, x.size), replace=False)
        for fi in flat_idx:
            idx = np.unravel_index(fi, x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            vp, vm = list(vals), list(vals)
            vp[pos], vm[pos] = xp, xm
            fd = (loss(vp) - loss(vm)) / (2 * h)
            ad = grads[n][idx]
            assert abs(fd - ad) <= 1e-6 * max(1.0, abs(ad)), (n, idx, fd, ad)
