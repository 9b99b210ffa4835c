"""Planted mistakes in the oracle must each be caught by at least one pin.

Each case copies the oracle's C++ source, applies one textual mutation (a dropped term, a wrong
sign or index, a transposed operand ...), compiles the copy on the CPU and runs the pin suite on
it.  The real oracle is never modified.
"""
import os
import tempfile

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "zeros_oracle.cpp")

MUTATIONS = [
    ("sigmoid sign", "1.0 / (1.0 + std::exp(-x))", "1.0 / (1.0 + std::exp(x))"),
    ("no normalisation", "y[a] = x[a] / n;", "y[a] = x[a];"),
    ("rotation sign", "x[a + half] = xa * s + xb * c;", "x[a + half] = -xa * s + xb * c;"),
    ("rotary frequency", "std::pow(base, -2.0 * a / d)", "std::pow(base, -1.0 * a / d)"),
    ("prior mean excludes token i",
     "        S[a] += ui[a];\n        ubar[a] = (et * mu[a] + S[a]) / (et + (i + 1));",
     "        ubar[a] = (et * mu[a] + S[a]) / (et + (i + 1));\n        S[a] += ui[a];"),
    ("prior weight", "ubar[a] = (et * mu[a] + S[a]) / (et + (i + 1));",
     "ubar[a] = (mu[a] + S[a]) / (et + (i + 1));"),
    ("logit scale", "s[i] = -dot / std::sqrt((double)d);\n  }\n}", "s[i] = -dot / d;\n  }\n}"),
    ("gamma drops sig_h/t",
     "const double gamma = -(sig1 - sigh) * P / (tcount * tcount) - sigh / tcount;",
     "const double gamma = -(sig1 - sigh) * P / (tcount * tcount);"),
    ("beta sign", "const double beta = (sig1 - sigh) / tcount;",
     "const double beta = (sigh - sig1) / tcount;"),
    ("transposed F update", "F[(size_t)a * d + j] += es * kv;", "F[(size_t)j * d + a] += es * kv;"),
    ("brute eps drops delta", "const double eps = soft - 1.0 / tc - delta / tc;\n      const double w_zs",
     "const double eps = soft - 1.0 / tc;\n      const double w_zs"),
    ("brute delta sign",
     "const double delta = s[i] - P / tc;\n      const double eps = soft - 1.0 / tc - delta / tc;"
     "\n      const double w_zs",
     "const double delta = P / tc - s[i];\n      const double eps = soft - 1.0 / tc - delta / tc;"
     "\n      const double w_zs"),
    ("encoder prior uses N+1", "ubar[a] = (et * mu[a] + S[a]) / (et + N);",
     "ubar[a] = (et * mu[a] + S[a]) / (et + N + 1);"),
    ("zero-order term dropped", "(gamma + zero_order) * Hs[e]", "gamma * Hs[e]"),
    ("zero-order over t+1", "sigmoid(pr.g0[base + t_idx]) / tcount",
     "sigmoid(pr.g0[base + t_idx]) / (tcount + 1)"),
    ("brute zero-order dropped", "const double w = w_zs + sig0 / tc;", "const double w = w_zs;"),
    ("layer norm unbiased variance", "    var /= d;", "    var /= (d - 1);"),
    ("layer norm eps outside sqrt", "1.0 / std::sqrt(var + eps)", "1.0 / (std::sqrt(var) + eps)"),
    ("layer norm head index", "const int h = (int)((r / N) % H);", "const int h = (int)(r % H);"),
    ("layer norm bias dropped", "* inv * gain + bias;", "* inv * gain;"),
    ("sm logit scale", "s[i] = dot / std::sqrt((double)d);", "s[i] = dot / d;"),
    ("sm delta without the mean",
     "const double delta = s[i] - P / tc;\n      const double eps = soft - 1.0 / tc - delta / tc;"
     "\n      const double w = sig1",
     "const double delta = s[i];\n      const double eps = soft - 1.0 / tc - delta / tc;"
     "\n      const double w = sig1"),
    ("sm eps drops delta", "const double eps = soft - 1.0 / tc - delta / tc;\n      const double w = sig1",
     "const double eps = soft - 1.0 / tc;\n      const double w = sig1"),
    ("sm rotary direction", "rotate(qr.data(), d, (double)(t - i), pr.rope_base);\n      double dot",
     "rotate(qr.data(), d, (double)(i - t), pr.rope_base);\n      double dot"),
    ("sm t off by one", "const int last = pr.causal ? t : N - 1;\n    const double tc = (double)(last + 1);\n    double m",
     "const int last = pr.causal ? t : N - 1;\n    const double tc = (double)(last + 2);\n    double m"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found or not unique: {name}"
    mutated = src.replace(old, new, 1)
    with tempfile.TemporaryDirectory() as tmp:
        cpp = os.path.join(tmp, "mut.cpp")
        with open(cpp, "w") as f:
            f.write(mutated)
        orc = oracle.Oracle(oracle.build(force=True, src=cpp, so=os.path.join(tmp, "mut.so")))
        caught = []
        for pin in oracle_pins.ALL_PINS:
            try:
                pin(orc)
            except AssertionError:
                caught.append(pin.__name__)
        assert caught, f"no pin catches the planted mistake: {name}"
