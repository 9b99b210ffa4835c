"""Fused output LayerNorm (each head's output row over its d columns) on every CUDA path vs the
fp64 oracle's forward followed by its LayerNorm (GPU only).

Tolerance.  The LayerNorm maps an output row o to (o - mean)/sqrt(var + eps) * w + b, whose
sensitivity to an error in o is |w| / sqrt(var + eps) for that row.  So the normalised error is
mapped back to the scale of o, |dy| / |w| * sqrt(var_ref + eps), and held to the forward's own
bound (tests/test_gpu_parity.py: over the compared outputs, relative to max|o_ref|, 1e-2 for
bf16 inputs with fp32 accumulation, 1e-5 for fp32; single-token sequences, whose exact output
is 0, in absolute terms).  A bf16 output adds its own rounding (2^-9
relative to |y|), which this back-mapping keeps below 2^-9 of the row's spread.
"""
import numpy as np
import pytest
import torch

import oracle
import zeros_inputs as zi
from tests.test_gpu_parity import TOL

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "u", "g1", "gh", "mu", "tau")


@pytest.fixture(scope="module")
def zs():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import zero_sum_prefix_gb300 as m
    m.load()
    return m


def _gain_bias(H, d, seed):
    gen = torch.Generator(device="cpu").manual_seed(seed)
    w = 1.0 + 0.5 * torch.rand((H, d), generator=gen)          # in [1, 1.5]: |w| >= 1
    b = 0.2 * torch.randn((H, d), generator=gen)
    return w.cuda(), b.cuda()


def ln_err(y, o_ref, w, b, eps):
    """Largest back-mapped LayerNorm error over every compared output, relative to max|o_ref|
    (absolute for single-token sequences, whose exact output is 0): the normalised error mapped
    back to the scale of o (divided by the gain, times the row's spread).  y, o_ref
    [B, H, N, d] numpy; w, b [H, d] numpy or None.  Also prints the worst single sequence."""
    y_ref = oracle.layer_norm(o_ref, w, b, eps)
    gain = np.ones(o_ref.shape[1:2] + o_ref.shape[3:]) if w is None else w
    spread = np.sqrt(np.var(o_ref, axis=-1, keepdims=True) + eps)      # [B, H, N, 1]
    back = np.abs(y - y_ref) / np.abs(gain)[None, :, None, :] * spread
    B, H, N, d = o_ref.shape
    if N == 1:
        err = float(back.max())
        print(f"back-mapped max abs error {err:.3e} (single token)")
        return err
    err = float(back.max() / np.abs(o_ref).max())
    per_seq = float((back.reshape(B * H, -1).max(axis=1) /
                     np.abs(o_ref).reshape(B * H, -1).max(axis=1)).max())
    print(f"back-mapped error {err:.3e} (worst single sequence {per_seq:.3e})")
    return err


def _run(zs, w, path, gain, eps, seed):
    inp = zi.make(w, "cuda")
    lw, lb = _gain_bias(w.H, w.d, seed) if gain else (None, None)
    args = [inp[n] for n in NAMES]
    y = zs.fwd(*args, causal=w.causal, rope=w.rope, rope_base=w.rope_base, path=path,
               ln=True, ln_w=lw, ln_b=lb, ln_eps=eps)
    o = zs.fwd(*args, causal=w.causal, rope=w.rope, rope_base=w.rope_base, path=path)
    assert zs.get_status() == 0
    return inp, y, o, lw, lb


@pytest.mark.parametrize("d,N,causal,dtype,path,gain,eps", [
    (64, 300, True, "bf16", "chunk", True, 1e-5), (128, 300, True, "bf16", "chunk", True, 1e-5),
    (64, 129, True, "bf16", "chunk", False, 1e-3), (128, 1, True, "bf16", "chunk", True, 1e-5),
    (64, 129, True, "bf16", "simt", True, 1e-5), (32, 77, True, "f32", "simt", True, 1e-5),
    (64, 77, True, "f32", "simt", True, 1e-5), (128, 40, True, "f32", "simt", False, 1e-5),
    (64, 50, False, "bf16", "simt", True, 1e-5), (128, 50, False, "f32", "simt", True, 1e-5),
    (64, 130, False, "f32", "auto", True, 1e-5), (64, 200, False, "bf16", "auto", False, 1e-5)])
def test_forward_layernorm(zs, d, N, causal, dtype, path, gain, eps):
    w = zi.Workload("ln", 2, 3, N, d, dtype=dtype, causal=causal, rope=causal,
                    seed=500 + d + N)
    inp, y, o, lw, lb = _run(zs, w, path, gain, eps, 7 + d)
    ref = oracle.forward(*(inp[n].cpu() for n in NAMES), causal=causal, rope=w.rope,
                         rope_base=w.rope_base)
    wn = None if lw is None else lw.cpu().double().numpy()
    bn = None if lb is None else lb.cpu().double().numpy()
    err = ln_err(y.float().cpu().double().numpy(), ref, wn, bn, eps)
    assert err <= TOL[dtype], err
    # with fp32 outputs the fused normalisation equals the same kernel's plain output
    # normalised afterwards (fp64), up to fp32 arithmetic
    if dtype == "f32":
        again = oracle.layer_norm(o.cpu().double().numpy(), wn, bn, eps)
        assert np.abs(y.cpu().double().numpy() - again).max() < 1e-4


def test_forward_layernorm_full_size_sampled(zs):
    """The bench's causal RoPE B8 H8 N4096 d64 bf16 launch with the LayerNorm: two sampled
    sequences against the oracle, every row of the batch normalised (mean 0 without bias)."""
    w = zi.CAUSAL_ROPE_B8H8N4096D64
    inp = zi.make(w, "cuda")
    lw, _ = _gain_bias(w.H, w.d, 77)
    args = [inp[n] for n in NAMES]
    y = zs.fwd(*args, causal=True, rope=True, rope_base=w.rope_base, ln=True, ln_w=lw)
    assert zs.get_status() == 0
    yf = y.float()
    # every row: sum_j y_j / w_j = 0 up to the bf16 rounding of each y_j (2^-9 relative)
    r = yf / lw[None, :, None, :]
    assert bool((r.sum(-1).abs() <= 2.0 ** -8 * r.abs().sum(-1) + 1e-3).all())
    for b, h in ((0, 0), (5, 6)):
        sel = {n: inp[n][b:b + 1, h:h + 1].cpu() for n in ("q", "k", "v", "u", "g1", "gh")}
        ref = oracle.forward(sel["q"], sel["k"], sel["v"], sel["u"], sel["g1"], sel["gh"],
                             inp["mu"][h:h + 1].cpu(), inp["tau"][h:h + 1].cpu(), causal=True,
                             rope=True, rope_base=w.rope_base)
        err = ln_err(yf[b:b + 1, h:h + 1].cpu().double().numpy(), ref,
                     lw[h:h + 1].cpu().double().numpy(), None, 1e-5)
        assert err <= TOL["bf16"], (b, h, err)


@pytest.mark.parametrize("d", [64, 128])
def test_decode_layernorm(zs, d):
    """Prefill, then decode steps with the LayerNorm; the state stays un-normalised."""
    B, H, N0, steps = 2, 2, 40, 6
    w = zi.Workload("lndec", B, H, N0, d, rope=True, seed=611 + d)
    pre = zi.make(w, "cuda")
    st = torch.empty(zs.state_bytes(B, H, d), dtype=torch.uint8, device="cuda")
    zs.fwd(*(pre[n] for n in NAMES), causal=True, rope=True, rope_base=w.rope_base,
           final_state=st)
    wf = w.with_(N=N0 + steps)
    full = zi.make(wf, "cuda")
    for n in ("q", "k", "v", "u", "g1", "gh"):
        full[n][:, :, :N0] = pre[n]
    full["mu"], full["tau"] = pre["mu"], pre["tau"]
    lw, lb = _gain_bias(H, d, 13)
    outs = []
    for t in range(N0, N0 + steps):
        outs.append(zs.decode_step(st, *(full[n][:, :, t].contiguous() for n in
                                         ("q", "k", "v", "u", "g1", "gh")),
                                   ln_w=lw, ln_b=lb, ln_eps=1e-5))
    assert zs.get_status() == 0
    ref = oracle.forward(*(full[n].cpu() for n in NAMES), causal=True, rope=True,
                         rope_base=w.rope_base)[:, :, N0:]
    dec = torch.stack(outs, dim=2).float().cpu().double().numpy()
    err = ln_err(dec, ref, lw.cpu().double().numpy(), lb.cpu().double().numpy(), 1e-5)
    assert err <= TOL["bf16"], err
