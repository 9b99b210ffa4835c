"""Writes tests/golden/two_token.json: hand-derivable two-token cases of the ZeroS layer.

No oracle code is used here.  Each case picks inputs whose deviation logits follow by hand from
the prior-mean definition (Paper-Notes "ZeroS: Zero-Sum Linear Attention for Efficient
Transformers", method details, "deviation logits"), then evaluates the two-token closed form
of the zero-sum weights derived from the softmax split of the same page ("zero-order removal
and zero-sum weights"):

  with Delta = s_1 - s_2, softmax_{2,1} = sigmoid(Delta), delta_{2,1} = Delta/2,
  eps_{2,1} = sigmoid(Delta) - 1/2 - Delta/4,
  w_{2,1} = sig1 * Delta/4 + sigh * (sigmoid(Delta) - 1/2 - Delta/4),  w_{2,2} = -w_{2,1},
  o_1 = 0,  o_2 = w_{2,1} (c_{2,1} v_1 - c_{2,2} v_2),

where c_{t,i} = q_hat_t R_{t-i} k_hat_i^T is the angular factor (radial-angular decoupling and
its RoPE form on the same page).  The page's motivating example is exactly this: two tokens,
where a convex combination can never produce v_1 - v_2 but a zero-sum weight can.

Run:  python tests/golden/make_golden.py   (needs mpmath, shipped with sympy)
"""
import json
import os

import mpmath as mp

mp.mp.dps = 50


def sig(x):
    return 1 / (1 + mp.e ** (-x))


def case_a():
    # d = 4, tau = 0 (e^tau = 1), mu = 0.
    # ubar_1 = u_1 / 2 = (1/2, 0, 0, 0)            -> s_1 = -(1 * 1/2) / sqrt(4) = -1/4
    # ubar_2 = (u_1 + u_2) / 3 = (1/3, 2/3, 0, 0)   -> s_2 = -(2 * 2/3) / 2 = -2/3
    # k_2 = 2 k_1, so k_hat_2 = k_hat_1 and c_{2,1} = c_{2,2} = q_hat_2 . k_hat_1 = 1/sqrt 2.
    s1, s2 = mp.mpf(-1) / 4, mp.mpf(-2) / 3
    g1 = [0.25, 0.5]
    gh = [-0.75, -0.3]
    q = [[0.0, 1.0, -1.0, 0.5], [1.0, 1.0, 0.0, 0.0]]
    k = [[1.0, 0.0, 0.0, 0.0], [2.0, 0.0, 0.0, 0.0]]
    v = [[1.0, 2.0, 3.0, 4.0], [0.0, -1.0, 5.0, 2.0]]
    u = [[1.0, 0.0, 0.0, 0.0], [0.0, 2.0, 0.0, 0.0]]
    c21 = c22 = 1 / mp.sqrt(2)
    return dict(name="two tokens, collinear keys, no rope", d=4, tau=0.0, mu=[0.0] * 4,
                rope=False, q=q, k=k, v=v, u=u, g1=g1, gh=gh, s=[s1, s2], c21=c21, c22=c22)


def case_b():
    # d = 2 (one rotary pair, theta_0 = base^0 = 1 for any base), tau = 0, mu = 0.
    # ubar_1 = (1/2, 0) -> s_1 = -(1/2)/sqrt 2 ;  ubar_2 = (1/3, 1/3) -> s_2 = -(1/3)/sqrt 2
    # q_hat_2 R_1 = (cos 1, sin 1); c_{2,1} = (cos 1, sin 1) . (0, 1) = sin 1;
    # c_{2,2} = q_hat_2 R_0 k_hat_2 = (1, 0) . (1, 0) = 1.
    s1, s2 = -mp.mpf(1) / 2 / mp.sqrt(2), -mp.mpf(1) / 3 / mp.sqrt(2)
    g1 = [1.5, -0.4]
    gh = [0.2, 0.9]
    q = [[0.3, -0.7], [2.0, 0.0]]
    k = [[0.0, 3.0], [0.5, 0.0]]
    v = [[1.0, -1.0], [2.0, 3.0]]
    u = [[1.0, 0.0], [0.0, 1.0]]
    return dict(name="two tokens, rotary positions 0 and 1", d=2, tau=0.0, mu=[0.0, 0.0],
                rope=True, q=q, k=k, v=v, u=u, g1=g1, gh=gh, s=[s1, s2], c21=mp.sin(1),
                c22=mp.mpf(1))


def finish(c):
    s1, s2 = c["s"]
    delta = s1 - s2
    sig1, sigh = sig(mp.mpf(c["g1"][1])), sig(mp.mpf(c["gh"][1]))
    w21 = sig1 * delta / 4 + sigh * (sig(delta) - mp.mpf(1) / 2 - delta / 4)
    o2 = [w21 * (c["c21"] * mp.mpf(a) - c["c22"] * mp.mpf(b)) for a, b in zip(c["v"][0],
                                                                                 c["v"][1])]
    out = {key: c[key] for key in ("name", "d", "tau", "mu", "rope", "q", "k", "v", "u", "g1",
                                    "gh")}
    out["expected_s"] = [float(s1), float(s2)]
    out["expected_w21"] = float(w21)
    out["expected_o"] = [[0.0] * c["d"], [float(x) for x in o2]]
    return out


def main():
    cases = [finish(case_a()), finish(case_b())]
    doc = {
        "source": "Paper-Notes 'ZeroS: Zero-Sum Linear Attention for Efficient Transformers', "
                  "method details: deviation logits, zero-sum weights, radial-angular "
                  "decoupling with RoPE; two-token motivating example in 'current pain points'",
        "derivation": "hand-derived logits + two-token closed form, evaluated with mpmath "
                      "at 50 digits by tests/golden/make_golden.py",
        "cases": cases,
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "two_token.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
