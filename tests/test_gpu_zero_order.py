"""Optional zero-order gate of a first layer (w_{t,i} gains sigmoid(g0_t)/t, encoder /N) on
every CUDA path vs the fp64 oracle (GPU only).  Same tolerance metric as
tests/test_gpu_parity.py."""
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


def _g0(w, seed, shape=None):
    gen = torch.Generator(device="cpu").manual_seed(seed)
    shape = shape or (w.B, w.H, w.N)
    return (torch.randn(shape, generator=gen, dtype=torch.float32) * 1.5).cuda()


def _oracle(inp, w, g0):
    args = [inp[n].cpu() for n in ("q", "k", "v", "u", "g1", "gh", "mu", "tau")]
    return oracle.forward(*args, causal=w.causal, rope=w.rope, rope_base=w.rope_base,
                          g0=g0.cpu())


@pytest.mark.parametrize("d,N,causal,dtype,path", [
    (64, 300, True, "bf16", "chunk"), (128, 300, True, "bf16", "chunk"),
    (64, 129, True, "bf16", "simt"), (32, 77, True, "f32", "simt"),
    (64, 50, False, "bf16", "simt"), (64, 50, False, "f32", "simt"),
    (64, 150, False, "bf16", "auto"), (64, 70, False, "f32", "auto")])
def test_forward_with_zero_order_gate(zs, d, N, causal, dtype, path):
    w = zi.Workload("g0", 2, 2, N, d, dtype=dtype, causal=causal, rope=causal, seed=300 + d + N)
    inp = zi.make(w, "cuda")
    g0 = _g0(w, 5 + N)
    args = [inp[n] for n in ("q", "k", "v", "u", "g1", "gh", "mu", "tau")]
    o = zs.fwd(*args, causal=causal, rope=w.rope, rope_base=w.rope_base, path=path, g0=g0)
    o_plain = zs.fwd(*args, causal=causal, rope=w.rope, rope_base=w.rope_base, path=path)
    assert zs.get_status() == 0
    ref = _oracle(inp, w, g0)
    S = w.B * w.H
    assert seq_err(o.float().cpu().numpy().reshape(S, N, d), ref.reshape(S, N, d)) <= TOL[dtype]
    # the gate really contributes (relative to the zero-sum output)
    diff = (o.float() - o_plain.float()).abs().max().item()
    assert diff > 10 * TOL[dtype] * o_plain.float().abs().max().item()


def test_decode_with_zero_order_gate(zs):
    """Prefill, then decode steps with the zero-order gate: outputs match the oracle over the
    whole sequence with the same gate."""
    B, H, d, N0, steps = 2, 2, 64, 40, 12
    w = zi.Workload("g0dec", B, H, N0, d, rope=True, seed=411)
    pre = zi.make(w, "cuda")
    st = torch.empty(zs.state_bytes(B, H, d), dtype=torch.uint8, device="cuda")
    zs.fwd(*(pre[n] for n in ("q", "k", "v", "u", "g1", "gh", "mu", "tau")), causal=True,
           rope=True, rope_base=w.rope_base, final_state=st)
    wf = w.with_(N=N0 + steps)
    full = zi.make(wf, "cuda")  # same seed: the first N0 tokens of a longer draw are not reused
    for n in ("q", "k", "v", "u", "g1", "gh"):
        full[n][:, :, :N0] = pre[n]
    full["mu"], full["tau"] = pre["mu"], pre["tau"]
    g0 = _g0(wf, 9)
    outs = []
    for t in range(N0, N0 + steps):
        o = zs.decode_step(st, *(full[n][:, :, t].contiguous() for n in
                                 ("q", "k", "v", "u", "g1", "gh")),
                           g0=g0[:, :, t].contiguous())
        outs.append(o)
    assert zs.get_status() == 0
    ref = _oracle(full, wf, g0)[:, :, N0:]
    dec = torch.stack(outs, dim=2).float().cpu().numpy()
    assert seq_err(dec.reshape(B * H, steps, d), ref.reshape(B * H, steps, d)) <= TOL["bf16"]
