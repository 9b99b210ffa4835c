"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

Every ``pin_*`` function takes an ``oracle.Oracle`` and raises ``AssertionError`` when the
oracle disagrees with the fact it checks.  ``tests/test_oracle_pins.py`` runs them on the real
oracle; ``tests/test_oracle_mutations.py`` runs them on deliberately broken copies of the
oracle to show that each plausible mistake is caught by at least one pin.

Sources of the facts (page titles and sections):
  * Paper-Notes "ZeroS: Zero-Sum Linear Attention for Efficient Transformers":
      - "current pain points": two tokens, v_1 - v_2 unreachable with convex weights;
      - method details / key design: zero-sum weights (sum_i w_{t,i} = 0), radial-angular
        decoupling with cos(theta) = q_hat k_hat^T and its RoPE form q_hat R_{t-i} k_hat^T,
        deviation logits with the prior-smoothed cumulative mean, linear-time prefix scan;
      - highlights: Lemma 3.4 norm bound.
  * ai.info AI summary, "Main Findings": Lemma 3.4, ||sum_i w_{t,i} v_i|| <= B t max_i|w_{t,i}|.
"""
from __future__ import annotations

import json
import os

import numpy as np
from scipy.special import softmax

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "two_token.json")


def rand_problem(seed, B=1, H=2, N=48, d=8, tau_range=1.0, gate_std=1.0):
    rng = np.random.default_rng(seed)
    q, k, v, u = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    g1 = rng.standard_normal((B, H, N)) * gate_std
    gh = rng.standard_normal((B, H, N)) * gate_std
    mu = rng.standard_normal((H, d))
    tau = rng.uniform(-tau_range, tau_range, H)
    return dict(q=q, k=k, v=v, u=u, g1=g1, gh=gh, mu=mu, tau=tau)


def relerr(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


def _args(p):
    return (p["q"], p["k"], p["v"], p["u"], p["g1"], p["gh"], p["mu"], p["tau"])


# ---------------------------------------------------------------------------------------------
def pin_golden_two_token(orc):
    """Hand-derived two-token cases (logits and outputs) from tests/golden/two_token.json."""
    with open(GOLDEN) as f:
        doc = json.load(f)
    for c in doc["cases"]:
        d = c["d"]
        shape4 = (1, 1, 2, d)
        p = dict(q=np.array(c["q"]).reshape(shape4), k=np.array(c["k"]).reshape(shape4),
                 v=np.array(c["v"]).reshape(shape4), u=np.array(c["u"]).reshape(shape4),
                 g1=np.array(c["g1"]).reshape(1, 1, 2), gh=np.array(c["gh"]).reshape(1, 1, 2),
                 mu=np.array(c["mu"]).reshape(1, d), tau=np.array([c["tau"]]))
        exp_o = np.array(c["expected_o"]).reshape(shape4)
        out, s, _, _ = orc.forward(*_args(p), causal=True, rope=c["rope"], debug=True)
        assert np.allclose(s.reshape(-1), c["expected_s"], rtol=0, atol=1e-14), c["name"]
        assert np.allclose(out, exp_o, rtol=0, atol=1e-14), c["name"]
        ob, _, wm = orc.brute(*_args(p), causal=True, rope=c["rope"])
        assert np.allclose(ob, exp_o, rtol=0, atol=1e-14), c["name"]
        assert abs(wm.reshape(-1)[1] - abs(c["expected_w21"])) < 1e-14, c["name"]


def pin_brute_vs_recurrent(orc):
    """The five-state recurrence equals the O(N^2) definition (exact algebra, fp64 rounding)."""
    for seed, (N, d) in enumerate([(1, 4), (2, 6), (33, 8), (64, 16)]):
        p = rand_problem(100 + seed, N=N, d=d)
        for causal in (True, False):
            for rope in (False, True):
                o = orc.forward(*_args(p), causal=causal, rope=rope)
                ob, _, _ = orc.brute(*_args(p), causal=causal, rope=rope)
                err = np.abs(o - ob).max() / max(np.abs(ob).max(), 1.0)
                assert err < 1e-12, (N, d, causal, rope, err)


def pin_zero_sum(orc):
    """sum_i w_{t,i} = 0 for every t, to 1e-12 (zero-order removal), causal and encoder."""
    p = rand_problem(7, N=256, d=32, H=1)
    for causal in (True, False):
        _, ws, wm = orc.brute(*_args(p), causal=causal)
        assert np.abs(ws).max() < 1e-12, np.abs(ws).max()
        assert wm.max() > 1e-6  # weights are not trivially zero


def pin_first_output_zero(orc):
    """o_1 = 0: one token has delta = 0 and softmax = 1 = 1/t, so w_{1,1} = 0."""
    p = rand_problem(8, N=16, d=8)
    ob, _, _ = orc.brute(*_args(p), causal=True)
    assert np.abs(ob[:, :, 0]).max() == 0.0
    o = orc.forward(*_args(p), causal=True)
    assert np.abs(o[:, :, 0]).max() <= 1e-12 * np.abs(o).max()


def pin_lemma_3_4(orc):
    """||o_t|| <= max_i ||v_i|| * t * max_i |w_{t,i}| (Lemma 3.4; |cos theta| <= 1)."""
    p = rand_problem(9, N=96, d=8, H=2)
    for causal in (True, False):
        o = orc.forward(*_args(p), causal=causal, rope=True)
        _, _, wm = orc.brute(*_args(p), causal=causal, rope=True)
        N = o.shape[2]
        vnorm = np.linalg.norm(p["v"], axis=-1)
        for b in range(o.shape[0]):
            for h in range(o.shape[1]):
                for t in range(N):
                    last = t if causal else N - 1
                    bound = vnorm[b, h, : last + 1].max() * (last + 1) * wm[b, h, t]
                    assert np.linalg.norm(o[b, h, t]) <= bound * (1 + 1e-12) + 1e-15


def pin_two_token_collinear(orc):
    """With k_2 = lambda k_1 (no rope), o_2 is a signed multiple of v_1 - v_2."""
    rng = np.random.default_rng(10)
    for _ in range(5):
        p = rand_problem(int(rng.integers(1 << 30)), N=2, d=6, H=1)
        p["k"][:, :, 1] = p["k"][:, :, 0] * rng.uniform(0.1, 3.0)
        o = orc.forward(*_args(p), causal=True)
        dv = (p["v"][0, 0, 0] - p["v"][0, 0, 1])
        o2 = o[0, 0, 1]
        resid = o2 - (o2 @ dv) / (dv @ dv) * dv
        assert np.linalg.norm(resid) <= 1e-13 * max(np.linalg.norm(o2), 1e-300)
        assert np.linalg.norm(o2) > 0


def pin_constant_logits(orc):
    """All u_j = mu = c 1: every logit is equal, delta = eps = 0, so o = 0."""
    p = rand_problem(11, N=40, d=8)
    c = 0.37
    p["u"][:] = c
    p["mu"][:] = c
    for causal in (True, False):
        o = orc.forward(*_args(p), causal=causal, rope=True)
        assert np.abs(o).max() < 1e-13


def _cos_matrix(p, b, h):
    qn = p["q"][b, h] / np.linalg.norm(p["q"][b, h], axis=-1, keepdims=True)
    kn = p["k"][b, h] / np.linalg.norm(p["k"][b, h], axis=-1, keepdims=True)
    return qn @ kn.T


def pin_equal_gates_softmax(orc):
    """sig1 = sigh = sig: w = sig (softmax - 1/t), i.e. softmax attention over the logits
    (scipy's textbook softmax) minus the uniform average, times cos(theta)."""
    p = rand_problem(12, N=50, d=8, H=2)
    p["gh"] = p["g1"].copy()
    for causal in (True, False):
        o, s, _, _ = orc.forward(*_args(p), causal=causal, debug=True)
        N = o.shape[2]
        for b in range(o.shape[0]):
            for h in range(o.shape[1]):
                C = _cos_matrix(p, b, h)
                for t in range(N):
                    last = t if causal else N - 1
                    sm = softmax(s[b, h, : last + 1])
                    w = (sm - 1.0 / (last + 1)) / (1 + np.exp(-p["g1"][b, h, t]))
                    ref = (w * C[t, : last + 1]) @ p["v"][b, h, : last + 1]
                    assert np.allclose(o[b, h, t], ref, rtol=0, atol=1e-13)


def _rope_rows(x, base):
    """Standard rotary embedding (Su et al., half-split pairs), row n at position n."""
    n, d = x.shape
    half = d // 2
    theta = base ** (-2.0 * np.arange(half) / d)
    ang = np.arange(n)[:, None] * theta[None, :]
    c, s = np.cos(ang), np.sin(ang)
    return np.concatenate([x[:, :half] * c - x[:, half:] * s, x[:, :half] * s + x[:, half:] * c],
                          axis=1)


def pin_equal_gates_softmax_rope(orc):
    """As pin_equal_gates_softmax, with cos(theta') = q_hat R_{t-i} k_hat^T from a textbook
    rotary embedding applied to the unit vectors at absolute positions."""
    p = rand_problem(19, N=40, d=16, H=1)
    p["gh"] = p["g1"].copy()
    base = 500.0
    o, s, _, _ = orc.forward(*_args(p), causal=True, rope=True, rope_base=base, debug=True)
    qn = p["q"][0, 0] / np.linalg.norm(p["q"][0, 0], axis=-1, keepdims=True)
    kn = p["k"][0, 0] / np.linalg.norm(p["k"][0, 0], axis=-1, keepdims=True)
    C = _rope_rows(qn, base) @ _rope_rows(kn, base).T
    for t in range(o.shape[2]):
        w = (softmax(s[0, 0, : t + 1]) - 1.0 / (t + 1)) / (1 + np.exp(-p["g1"][0, 0, t]))
        ref = (w * C[t, : t + 1]) @ p["v"][0, 0, : t + 1]
        assert np.allclose(o[0, 0, t], ref, rtol=0, atol=1e-13)


def pin_linear_gate_limit(orc):
    """sigh -> 0 (gh = -40): o_t = (sig1/t) sum_i (s_i - mean s) cos(theta) v_i."""
    p = rand_problem(13, N=40, d=8, H=1)
    p["gh"][:] = -40.0
    o, s, _, _ = orc.forward(*_args(p), causal=True, debug=True)
    C = _cos_matrix(p, 0, 0)
    for t in range(o.shape[2]):
        st = s[0, 0, : t + 1]
        w = (st - st.mean()) / (t + 1) / (1 + np.exp(-p["g1"][0, 0, t]))
        ref = (w * C[t, : t + 1]) @ p["v"][0, 0, : t + 1]
        assert np.allclose(o[0, 0, t], ref, rtol=0, atol=1e-13)


def pin_rope_relative(orc):
    """Only relative positions matter: shifting every rotary position leaves o unchanged."""
    p = rand_problem(14, N=30, d=8)
    for causal in (True, False):
        a = orc.forward(*_args(p), causal=causal, rope=True, pos0=0.0)
        b = orc.forward(*_args(p), causal=causal, rope=True, pos0=1234.0)
        assert relerr(a, b) < 1e-10


def pin_scale_and_linearity(orc):
    """q and k enter only through their directions; o is linear in v."""
    p = rand_problem(15, N=24, d=8)
    base = orc.forward(*_args(p), causal=True, rope=True)
    p2 = dict(p)
    p2["q"] = p["q"] * 3.5
    p2["k"] = p["k"] * np.linspace(0.2, 4.0, p["k"].shape[2])[None, None, :, None]
    assert relerr(orc.forward(*_args(p2), causal=True, rope=True), base) < 1e-12
    rng = np.random.default_rng(16)
    v2 = rng.standard_normal(p["v"].shape)
    p3 = dict(p)
    p3["v"] = 2.0 * p["v"] - v2
    p4 = dict(p)
    p4["v"] = v2
    comb = orc.forward(*_args(p3), causal=True, rope=True)
    ref = 2.0 * base - orc.forward(*_args(p4), causal=True, rope=True)
    assert relerr(comb, ref) < 1e-12


def pin_prior_limits(orc):
    """tau -> +inf gives ubar_i = mu; tau -> -inf gives the plain cumulative mean."""
    p = rand_problem(17, N=20, d=8, H=1)
    d = p["u"].shape[-1]
    u = p["u"][0, 0]
    p["tau"][:] = 40.0
    _, s, _, _ = orc.forward(*_args(p), causal=True, debug=True)
    ref = -(u @ p["mu"][0]) / np.sqrt(d)
    assert np.allclose(s[0, 0], ref, rtol=1e-12, atol=1e-12)
    p["tau"][:] = -40.0
    _, s, _, _ = orc.forward(*_args(p), causal=True, debug=True)
    cmean = np.cumsum(u, axis=0) / np.arange(1, u.shape[0] + 1)[:, None]
    ref = -np.einsum("ia,ia->i", u, cmean) / np.sqrt(d)
    assert np.allclose(s[0, 0], ref, rtol=1e-12, atol=1e-12)


def pin_prefix_sums(orc):
    """E_t and P_t reported by the recurrence are the prefix sums of e^{s_i} and s_i."""
    p = rand_problem(18, N=30, d=8)
    _, s, E, P = orc.forward(*_args(p), causal=True, debug=True)
    assert np.allclose(E, np.cumsum(np.exp(s), axis=-1), rtol=1e-13)
    assert np.allclose(P, np.cumsum(s, axis=-1), rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------------------------------
# Zero-order gate of a first layer (Paper-Notes, zero-order removal: "the first layer may keep
# the zero-order term"; ai.info: "optionally sigma^0_t in the first layer"): w_{t,i} gains
# sig^0_t / t.

def _sig(x):
    return 1.0 / (1.0 + np.exp(-x))


def _uniform_angular(p, b, h, t, last, rope, base, g0):
    """sig^0_t/(last+1) * sum_{i<=last} cos(theta_{t,i}) v_i, with a textbook rotary map."""
    qn = p["q"][b, h] / np.linalg.norm(p["q"][b, h], axis=-1, keepdims=True)
    kn = p["k"][b, h] / np.linalg.norm(p["k"][b, h], axis=-1, keepdims=True)
    if rope:
        qn, kn = _rope_rows(qn, base), _rope_rows(kn, base)
    c = qn[t] @ kn[: last + 1].T
    return _sig(g0[b, h, t]) / (last + 1) * (c @ p["v"][b, h, : last + 1])


def pin_zero_order_sum(orc):
    """With the zero-order gate the weights sum to sig^0_t (not 0), and the five-state form
    still equals the definition."""
    p = rand_problem(21, N=64, d=8, H=2)
    g0 = np.random.default_rng(22).standard_normal(p["g1"].shape) * 2.0
    for causal in (True, False):
        for rope in (False, True):
            o = orc.forward(*_args(p), causal=causal, rope=rope, g0=g0)
            ob, ws, _ = orc.brute(*_args(p), causal=causal, rope=rope, g0=g0)
            assert np.abs(ws - _sig(g0)).max() < 1e-12
            assert np.abs(o - ob).max() / max(np.abs(ob).max(), 1.0) < 1e-12


def pin_zero_order_uniform(orc):
    """sig^1 = sig^h = 0 (gate logits -1000): only the zero-order term is left, the uniform
    average of the angular-weighted values: o_t = (sig^0_t / t) sum_{i<=t} cos(theta) v_i."""
    p = rand_problem(23, N=30, d=8, H=2)
    p["g1"][:] = -1000.0
    p["gh"][:] = -1000.0
    g0 = np.random.default_rng(24).standard_normal(p["g1"].shape)
    base = 300.0
    for causal in (True, False):
        for rope in (False, True):
            o = orc.forward(*_args(p), causal=causal, rope=rope, rope_base=base, g0=g0)
            N = o.shape[2]
            for b in range(o.shape[0]):
                for h in range(o.shape[1]):
                    for t in range(N):
                        last = t if causal else N - 1
                        ref = _uniform_angular(p, b, h, t, last, rope, base, g0)
                        assert np.allclose(o[b, h, t], ref, rtol=0, atol=1e-13)


def pin_zero_order_linearity(orc):
    """The zero-order term adds (sig^0_t / t) sum_{i<=t} cos(theta) v_i to the zero-sum output."""
    p = rand_problem(25, N=24, d=8, H=1)
    g0 = np.random.default_rng(26).standard_normal(p["g1"].shape)
    for causal in (True, False):
        o0 = orc.forward(*_args(p), causal=causal, rope=True)
        o1 = orc.forward(*_args(p), causal=causal, rope=True, g0=g0)
        N = o0.shape[2]
        for t in range(N):
            last = t if causal else N - 1
            ref = _uniform_angular(p, 0, 0, t, last, True, 10000.0, g0)
            assert np.allclose(o1[0, 0, t] - o0[0, 0, t], ref, rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------------------------
# Output LayerNorm (Paper-Notes, ablation table "without LayerNorm" and the highlights' remark that
# LayerNorm supersedes the 1/sqrt(t) Lipschitz decay; placement read as each head's output row).
def _ln_params(seed, H, d):
    rng = np.random.default_rng(seed)
    return 1.0 + 0.5 * rng.standard_normal((H, d)), 0.3 * rng.standard_normal((H, d))


def pin_layer_norm_moments(orc):
    """Without gain and bias every normalised row has mean 0 and population variance
    var / (var + eps), var being the row's own population variance (numpy)."""
    p = rand_problem(31, B=2, H=3, N=20, d=16)
    o = orc.forward(*_args(p), causal=True, rope=True)
    for eps in (1e-5, 0.25):
        y = orc.layer_norm(o, eps=eps)
        var = np.var(o, axis=-1)
        assert np.abs(y.mean(-1)).max() < 1e-13
        rows = var > 0
        assert np.allclose(np.var(y, axis=-1)[rows], (var / (var + eps))[rows], rtol=1e-12, atol=0)


def pin_layer_norm_library(orc):
    """Gain and bias per head: every head's rows equal torch.nn.functional.layer_norm (fp64)."""
    import torch
    p = rand_problem(32, B=2, H=3, N=17, d=8)
    w, b = _ln_params(33, 3, 8)
    for causal in (True, False):
        o = orc.forward(*_args(p), causal=causal, rope=False)
        y = orc.layer_norm(o, w, b, eps=1e-5)
        for h in range(3):
            ref = torch.nn.functional.layer_norm(torch.from_numpy(o[:, h]), (8,),
                                                 torch.from_numpy(w[h]), torch.from_numpy(b[h]),
                                                 eps=1e-5).numpy()
            assert np.allclose(y[:, h], ref, rtol=0, atol=1e-12)


def pin_layer_norm_first_row(orc):
    """The first causal output is zero (the one weight of a single token is zero; the recurrence
    leaves rounding residue near 1e-16), so its normalised row is the head's bias."""
    p = rand_problem(34, B=1, H=2, N=5, d=8)
    w, b = _ln_params(35, 2, 8)
    y = orc.layer_norm(orc.forward(*_args(p), causal=True), w, b, eps=1e-5)
    assert np.allclose(y[:, :, 0], np.broadcast_to(b, y[:, :, 0].shape), rtol=0, atol=1e-9)
    assert not np.allclose(y[:, :, 1], np.broadcast_to(b, y[:, :, 1].shape), rtol=0, atol=1e-3)


# ---------------------------------------------------------------------------------------------
# ZeroS-SM: the zero-sum reweighting of standard softmax attention (Paper-Notes, linear-time
# prefix scan: "the same reweighting can be applied to standard softmax attention"; the
# two-token contrast v_1 - v_2 of the "current pain points" section).
def _sm_args(p):
    return (p["q"], p["k"], p["v"], p["g1"], p["gh"])


def _logistic(x):
    return 1.0 / (1.0 + np.exp(-x))


def pin_sm_two_token(orc):
    """Closed form for two tokens: with D = s_{2,1} - s_{2,2}, w_{2,1} = sig1 D/4 +
    sigh (logistic(D) - 1/2 - D/4) = -w_{2,2}, so o_2 = w_{2,1} (v_1 - v_2); and o_1 = 0."""
    for seed, rope in ((41, False), (42, True)):
        p = rand_problem(seed, B=1, H=3, N=2, d=8)
        o = orc.sm(*_sm_args(p), causal=True, rope=rope, rope_base=100.0)
        for h in range(3):
            q, k, v = p["q"][0, h], p["k"][0, h], p["v"][0, h]
            if rope:
                q, k = _rope_rows(q, 100.0), _rope_rows(k, 100.0)
            D = (q[1] @ k[0] - q[1] @ k[1]) / np.sqrt(8)
            s1, sh = _logistic(p["g1"][0, h, 1]), _logistic(p["gh"][0, h, 1])
            w21 = s1 * D / 4 + sh * (_logistic(D) - 0.5 - D / 4)
            assert np.allclose(o[0, h, 1], w21 * (v[0] - v[1]), rtol=0, atol=1e-14)
            assert np.abs(o[0, h, 0]).max() < 1e-15


def pin_sm_equal_gates_softmax(orc):
    """sig1 = sigh = sig: w = sig (softmax - 1/t): scipy's softmax attention over the masked
    logits Q K^T / sqrt d (textbook rotary map with rope) minus the mean of the values."""
    for causal, rope in ((True, False), (False, False), (True, True)):
        p = rand_problem(43, B=1, H=2, N=30, d=8)
        p["gh"] = p["g1"].copy()
        o = orc.sm(*_sm_args(p), causal=causal, rope=rope, rope_base=300.0)
        N = o.shape[2]
        for h in range(2):
            q, k, v = p["q"][0, h], p["k"][0, h], p["v"][0, h]
            if rope:
                q, k = _rope_rows(q, 300.0), _rope_rows(k, 300.0)
            S = q @ k.T / np.sqrt(8)
            for t in range(N):
                last = t if causal else N - 1
                att = softmax(S[t, : last + 1]) @ v[: last + 1]
                ref = _logistic(p["g1"][0, h, t]) * (att - v[: last + 1].mean(axis=0))
                assert np.allclose(o[0, h, t], ref, rtol=0, atol=1e-13)


def pin_sm_linear_gate_limit(orc):
    """sigh -> 0: o_t = (sig1/t) sum_i (s_{t,i} - mean_i s_{t,i}) v_i, the centred logits as
    weights of a linear attention (numpy matrix products)."""
    p = rand_problem(44, B=1, H=1, N=25, d=8)
    p["gh"][:] = -40.0
    o = orc.sm(*_sm_args(p), causal=True)
    S = p["q"][0, 0] @ p["k"][0, 0].T / np.sqrt(8)
    for t in range(25):
        st = S[t, : t + 1]
        w = _logistic(p["g1"][0, 0, t]) * (st - st.mean()) / (t + 1)
        assert np.allclose(o[0, 0, t], w @ p["v"][0, 0, : t + 1], rtol=0, atol=1e-13)


def pin_sm_zero_sum_and_shift(orc):
    """The weights of every query sum to zero (plus sig0 with the zero-order gate); adding one
    vector to every key shifts a query's logits by a constant, which changes nothing."""
    p = rand_problem(45, B=2, H=2, N=20, d=8)
    g0 = np.random.default_rng(46).standard_normal(p["g1"].shape)
    for causal in (True, False):
        _, ws = orc.sm(*_sm_args(p), causal=causal, wsum=True)
        assert np.abs(ws).max() < 1e-13
        _, ws0 = orc.sm(*_sm_args(p), causal=causal, wsum=True, g0=g0)
        assert np.allclose(ws0, _logistic(g0), rtol=0, atol=1e-13)
        a = orc.sm(*_sm_args(p), causal=causal)
        p2 = dict(p, k=p["k"] + np.random.default_rng(47).standard_normal(8))
        b = orc.sm(*_sm_args(p2), causal=causal)
        assert relerr(b, a) < 1e-10


ALL_PINS = [pin_golden_two_token, pin_brute_vs_recurrent, pin_zero_sum, pin_first_output_zero,
            pin_lemma_3_4, pin_two_token_collinear, pin_constant_logits, pin_equal_gates_softmax,
            pin_equal_gates_softmax_rope, pin_linear_gate_limit, pin_rope_relative, pin_scale_and_linearity, pin_prior_limits,
            pin_prefix_sums,
            pin_zero_order_sum, pin_zero_order_uniform, pin_zero_order_linearity,
            pin_layer_norm_moments, pin_layer_norm_library, pin_layer_norm_first_row,
            pin_sm_two_token, pin_sm_equal_gates_softmax, pin_sm_linear_gate_limit,
            pin_sm_zero_sum_and_shift]
