"""ZeroS-SM (the zero-sum reweighting of standard softmax attention) on the tensor-core kernel
vs the fp64 oracle (GPU only).

Tolerance: the metric of tests/test_gpu_parity.py (max error over max|o_ref| of the compared
outputs; single-token sequences, whose exact output is 0, in absolute terms) at the bf16 bound
1e-2.  The
kernel's error sources are the bf16 rounding of the weight tile W (once per weight, 2^-9
relative, after the three nearly cancelling terms were summed in fp32), of the rotated q and k
(rope), and of the output; products and sums are fp32.
"""
import numpy as np
import pytest
import torch

import oracle
import zeros_inputs as zi
from tests.test_gpu_parity import TOL, seq_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zs():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import zero_sum_prefix_gb300 as m
    m.load()
    return m


def _inputs(B, H, N, d, seed):
    w = zi.Workload("sm", B, H, N, d, seed=seed)
    inp = zi.make(w, "cuda")
    return {n: inp[n] for n in ("q", "k", "v", "g1", "gh")}


def _g0(shape, seed):
    gen = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(shape, generator=gen) * 1.5).cuda()


@pytest.mark.parametrize("d,N,causal,rope,gate0", [
    (64, 300, True, False, False), (64, 300, True, True, False), (128, 300, True, True, False),
    (64, 1, True, False, False), (64, 128, True, False, True), (128, 129, True, False, False),
    (64, 200, False, False, False), (128, 77, False, True, True), (64, 513, True, True, True)])
def test_sm_parity(zs, d, N, causal, rope, gate0):
    B, H = 2, 2
    x = _inputs(B, H, N, d, 900 + d + N)
    g0 = _g0((B, H, N), 5) if gate0 else None
    o = zs.sm_fwd(x["q"], x["k"], x["v"], x["g1"], x["gh"], causal=causal, rope=rope,
                  rope_base=10000.0, g0=g0)
    assert zs.get_status() == 0
    ref = oracle.sm(*(x[n].cpu() for n in ("q", "k", "v", "g1", "gh")), causal=causal,
                    rope=rope, rope_base=10000.0, g0=None if g0 is None else g0.cpu())
    err = seq_err(o.float().cpu().numpy().reshape(B * H, N, d), ref.reshape(B * H, N, d))
    assert err <= TOL["bf16"], err


def test_sm_full_size(zs):
    """B8 H8 N4096 d64, causal: two sampled sequences against the oracle, and for the whole
    batch the zero-sum property: with every value row equal to c (|c| <= 1), o_t =
    sum_i w_{t,i} c = 0 up to the bf16 rounding of each weight, |o_t| <= 2^-9 sum_i |w_{t,i}|;
    with logits of unit scale sum_i |w_{t,i}| is about 4 (sigh (1 + 1 + mean|delta|) +
    sig1 mean|delta|), so the bound 2e-2 leaves a margin of five."""
    B, H, N, d = 8, 8, 4096, 64
    x = _inputs(B, H, N, d, 4242)
    o = zs.sm_fwd(x["q"], x["k"], x["v"], x["g1"], x["gh"], causal=True)
    assert zs.get_status() == 0
    for b, h in ((0, 0), (7, 5)):
        ref = oracle.sm(*(x[n][b:b + 1, h:h + 1].cpu() for n in ("q", "k", "v", "g1", "gh")),
                        causal=True)
        err = seq_err(o[b:b + 1, h:h + 1].float().cpu().numpy().reshape(1, N, d),
                      ref.reshape(1, N, d))
        assert err <= TOL["bf16"], (b, h, err)
    c = torch.linspace(-1.0, 1.0, d, device="cuda").to(torch.bfloat16)
    vc = c.expand(B, H, N, d).contiguous()
    oc = zs.sm_fwd(x["q"], x["k"], vc, x["g1"], x["gh"], causal=True)
    assert zs.get_status() == 0
    assert oc.float().abs().max().item() < 2e-2


@pytest.mark.parametrize("causal,rope,gate0,N", [
    (True, True, False, 300), (True, False, True, 257), (False, True, True, 300),
    (False, False, False, 129)])
def test_sm_many_query_tiles_per_cta(zs, causal, rope, gate0, N):
    """d = 64 with more query tiles than CTAs (B8 H16: 256 to 384 tiles of 128 queries), so that
    each CTA of the d = 64 kernel takes several of them, of different key-tile counts, in a row:
    every sequence against the oracle."""
    B, H, d = 8, 16, 64
    x = _inputs(B, H, N, d, 3100 + N)
    g0 = _g0((B, H, N), 31) if gate0 else None
    o = zs.sm_fwd(x["q"], x["k"], x["v"], x["g1"], x["gh"], causal=causal, rope=rope,
                  rope_base=10000.0, g0=g0)
    assert zs.get_status() == 0
    ref = oracle.sm(*(x[n].cpu() for n in ("q", "k", "v", "g1", "gh")), causal=causal,
                    rope=rope, rope_base=10000.0, g0=None if g0 is None else g0.cpu())
    err = seq_err(o.float().cpu().numpy().reshape(B * H, N, d), ref.reshape(B * H, N, d))
    assert err <= TOL["bf16"], err


def test_sm_zero_order_gate_constant_values(zs):
    """With the zero-order gate the weights of query t sum to sig0_t: constant values c give
    o_t = sig0_t c."""
    B, H, N, d = 2, 4, 700, 128
    x = _inputs(B, H, N, d, 77)
    g0 = _g0((B, H, N), 78)
    c = torch.linspace(-1.0, 1.0, d, device="cuda").to(torch.bfloat16)
    vc = c.expand(B, H, N, d).contiguous()
    for causal in (True, False):
        o = zs.sm_fwd(x["q"], x["k"], vc, x["g1"], x["gh"], causal=causal, g0=g0)
        assert zs.get_status() == 0
        ref = torch.sigmoid(g0)[..., None] * c.float()
        assert (o.float() - ref).abs().max().item() < 2e-2
