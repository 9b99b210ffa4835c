"""The seeded input generators (CPU): shapes, dtypes, determinism and the recipe's
distributions, at reduced sizes of every workload."""
import pytest
import torch

import zeros_inputs as zi


@pytest.mark.parametrize("w", zi.ALL, ids=lambda w: w.name)
def test_shapes_dtypes_and_determinism(w):
    B, N = 1, 64
    a = zi.make(w, "cpu", N=N, B=B)
    b = zi.make(w, "cpu", N=N, B=B)
    sd = zi.storage_dtype(w)
    for n in ("q", "k", "v", "u"):
        assert a[n].shape == (B, w.H, N, w.d) and a[n].dtype == sd and a[n].is_contiguous()
    for n in ("g1", "gh"):
        assert a[n].shape == (B, w.H, N) and a[n].dtype == torch.float32
    assert a["mu"].shape == (w.H, w.d) and a["tau"].shape == (w.H,)
    for n in a:
        assert torch.equal(a[n], b[n]), n  # same seed, same tensors
    other = zi.make(w.with_(seed=w.seed + 1), "cpu", N=N, B=B)
    assert not torch.equal(a["q"], other["q"])


def test_recipe_distributions():
    w = zi.CAUSAL_ROPE_B8H8N4096D64
    x = zi.make(w, "cpu", N=512, B=2)
    for n in ("q", "k", "v", "u"):
        t = x[n].float()
        assert abs(float(t.mean())) < 0.02 and abs(float(t.std()) - 1.0) < 0.02, n
    assert abs(float(x["g1"].std()) - w.gate_var ** 0.5) < 0.05
    assert float(x["tau"].abs().max()) <= 1.0
    # fixed tau
    f = zi.make(zi.CAUSAL_F32_SMALL, "cpu")
    assert torch.all(f["tau"] == 0.0)
    # the long-context workload scales every token's u row by one c in [0.5, 2]: its spread of
    # row norms is wider than the unscaled draw's
    lw = zi.LONG_ROPE_B2H16N65536D128
    lo = zi.make(lw, "cpu", N=256, B=1)["u"].float().norm(dim=-1)
    ref = zi.make(lw.with_(u_scale=None), "cpu", N=256, B=1)["u"].float().norm(dim=-1)
    assert float(lo.std() / lo.mean()) > 2.0 * float(ref.std() / ref.mean())
    assert abs(float(lw.gate_var) - 2.0) < 1e-12


def test_decode_tokens_and_sampled_heads():
    w = zi.DECODE_B256H32D128
    t0, t1 = zi.decode_tokens(w, 0), zi.decode_tokens(w, 1)
    for n in ("q", "k", "v", "u"):
        assert t0[n].shape == (w.B, w.H, w.d)
    assert t0["g1"].shape == (w.B, w.H)
    assert not torch.equal(t0["q"], t1["q"])  # a new draw per step
    assert torch.equal(t0["q"], zi.decode_tokens(w, 0)["q"])
    heads = zi.sample_heads(zi.CAUSAL_ROPE_B8H8N4096D64, 6)
    assert len(heads) == len(set(heads)) == 6 and heads == sorted(heads)
    assert all(0 <= b < 8 and 0 <= h < 8 for b, h in heads)
    assert len(zi.sample_heads(zi.CAUSAL_F32_SMALL, 10)) == 1
