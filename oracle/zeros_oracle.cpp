// ZeroS oracle: plain, slow, fp64 CPU reference of the zero-sum linear attention layer.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or calls this
// file; only the tests, the smoke check and the CPU-baseline leg of the benchmark use it.
// It shares no code, header, table or constant with the CUDA path.
//
// Sources (the method is described only in prose/LaTeX on these pages):
//   [PN]  "ZeroS: Zero-Sum Linear Attention for Efficient Transformers", Paper-Notes
//         (zhaoyang97.github.io, NeurIPS 2025 / llm_efficiency), section "方法详解" (method
//         details): "关键设计" (key design) -> zero-order removal / zero-sum weights,
//         radial-angular decoupling (+ RoPE), deviation logits, linear-time prefix scan;
//         "损失函数 / 训练策略" (causal and non-causal modes).
//   [AI]  ai.info AI summary of the same paper, "Methodology in Plain English" and
//         "Main Findings" (Lemma 3.4 norm bound).
//
// Two independent evaluations are provided:
//   zs_oracle_fwd   - the recurrent form with the five prefix states E, P, F, G, H ([PN],
//                     "linear-time prefix scan"); RoPE applied with absolute positions.
//   zs_oracle_brute - the O(N^2) definition: every weight w_{t,i} and every angular factor
//                     cos(theta_{t,i}) is materialised; RoPE applied as the relative rotation
//                     R_{t-i} ([PN], "radial-angular decoupling").
//
// Readings where the pages are silent:
//   * delta_{t,i} = s_i - P_t/t (first-order Taylor term of softmax about the mean logit) and
//     eps_{t,i} = softmax_{t,i} - 1/t - delta_{t,i}/t (the remainder).
//   * alpha_t = sig^h_t/E_t, beta_t = (sig^1_t - sig^h_t)/t,
//     gamma_t = -(sig^1_t - sig^h_t) P_t/t^2 - sig^h_t/t   (expansion of w in the three states).
//   * x_hat = x / max(||x||_2, 1e-12).
//   * RoPE: half-split pairs (a, a + d/2), theta_a = base^(-2a/d), position of token t is
//     t - 1 + pos0; rotation applied to the unit vectors.
//   * Encoder (non-causal) mode: every sum runs over all N tokens and t := N in delta, eps and
//     the coefficients; the prior mean is the full-sequence mean for every token.  Gates stay
//     per token.
//   * Zero-order gate (optional, first layer; [PN] zero-order removal: "the first layer may keep
//     the zero-order term"; [AI] "optionally sigma^0_t in the first layer"): the weight gains
//     the zero-order term itself, w_{t,i} += sig^0_t / t with sig^0_t = sigmoid(g0_t), so the
//     weights sum to sig^0_t; in the five-state form gamma_t gains sig^0_t / t.
//   * Output LayerNorm (optional; [PN] ablation table "without LayerNorm" and the Lipschitz
//     discussion of the highlights section name a LayerNorm on the layer's output but not its
//     placement): applied to each head's output row o_t over its d channels,
//     y = (o_t - mean) / sqrt(var + eps) * w + b with the biased variance, w and b per head
//     [H,d] (absent: 1 and 0).
//
//   * ZeroS-SM (quadratic variant): see sm_one.
//
// Parity pins for everything here live in tests/test_oracle_pins.py.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <thread>
#include <vector>

namespace {

struct Problem {
  const double *q, *k, *v, *u, *g1, *gh, *mu, *tau;
  const double* g0;  // nullable: zero-order gate logits [B,H,N]
  int B, H, N, d;
  int causal, rope;
  double rope_base;
  double pos0;
};

inline double sigmoid(double x) { return 1.0 / (1.0 + std::exp(-x)); }

// Unit-normalised copy of a row vector ([PN] radial-angular decoupling: q_hat, k_hat).
void unit_vector(const double* x, int d, double* y) {
  double ss = 0.0;
  for (int a = 0; a < d; ++a) ss += x[a] * x[a];
  const double n = std::max(std::sqrt(ss), 1e-12);
  for (int a = 0; a < d; ++a) y[a] = x[a] / n;
}

// Right-multiplication of a row vector by the rotary matrix R_p (angle p * theta_a on the
// pair (a, a + d/2)).  R_p R_{p'}^T = R_{p - p'}, which is how the relative form
// q_hat R_{t-i} k_hat^T of [PN] arises from absolute rotations.
void rotate(double* x, int d, double p, double base) {
  const int half = d / 2;
  for (int a = 0; a < half; ++a) {
    const double theta = std::pow(base, -2.0 * a / d);
    const double c = std::cos(p * theta), s = std::sin(p * theta);
    const double xa = x[a], xb = x[a + half];
    x[a] = xa * c - xb * s;
    x[a + half] = xa * s + xb * c;
  }
}

// Deviation logits s_i = -(1/sqrt d) u_i . ubar_i with the prior-smoothed cumulative mean
// ubar_i = (e^tau mu + sum_{j<=i} u_j) / (e^tau + i)   ([PN] "deviation logits").
// Encoder mode: ubar is the full-sequence mean for every i (reading, see header).
void deviation_logits(const double* u, const double* mu, double tau, int N, int d, int causal,
                      double* s) {
  const double et = std::exp(tau);
  std::vector<double> S(d, 0.0), ubar(d);
  if (!causal) {
    for (int i = 0; i < N; ++i)
      for (int a = 0; a < d; ++a) S[a] += u[(size_t)i * d + a];
    for (int a = 0; a < d; ++a) ubar[a] = (et * mu[a] + S[a]) / (et + N);
  }
  for (int i = 0; i < N; ++i) {
    const double* ui = u + (size_t)i * d;
    if (causal) {
      for (int a = 0; a < d; ++a) {
        S[a] += ui[a];
        ubar[a] = (et * mu[a] + S[a]) / (et + (i + 1));
      }
    }
    double dot = 0.0;
    for (int a = 0; a < d; ++a) dot += ui[a] * ubar[a];
    s[i] = -dot / std::sqrt((double)d);
  }
}

// Recurrent evaluation for one (b, h) sequence: the five prefix states of [PN]
// "linear-time prefix scan", E = sum e^s, P = sum s, F = sum e^s k^T v, G = sum s k^T v,
// H = sum k^T v, and o_t = q_hat_t (alpha_t F_t + beta_t G_t + gamma_t H_t).
void recurrent_one(const Problem& pr, int b, int h, double* out, double* dbg_s, double* dbg_E,
                   double* dbg_P) {
  const int N = pr.N, d = pr.d;
  const size_t base = ((size_t)b * pr.H + h) * (size_t)N;
  const double* q = pr.q + base * d;
  const double* k = pr.k + base * d;
  const double* v = pr.v + base * d;
  const double* u = pr.u + base * d;
  const double* g1 = pr.g1 + base;
  const double* gh = pr.gh + base;
  double* o = out + base * d;

  std::vector<double> s(N);
  deviation_logits(u, pr.mu + (size_t)h * d, pr.tau[h], N, d, pr.causal, s.data());

  std::vector<double> F((size_t)d * d, 0.0), G((size_t)d * d, 0.0), Hs((size_t)d * d, 0.0);
  std::vector<double> qh(d), kh(d);
  double E = 0.0, P = 0.0;

  auto accumulate = [&](int i) {
    const double es = std::exp(s[i]);
    E += es;
    P += s[i];
    unit_vector(k + (size_t)i * d, d, kh.data());
    if (pr.rope) rotate(kh.data(), d, pr.pos0 + i, pr.rope_base);
    const double* vi = v + (size_t)i * d;
    for (int a = 0; a < d; ++a)
      for (int j = 0; j < d; ++j) {
        const double kv = kh[a] * vi[j];
        F[(size_t)a * d + j] += es * kv;
        G[(size_t)a * d + j] += s[i] * kv;
        Hs[(size_t)a * d + j] += kv;
      }
  };
  auto readout = [&](int t_idx, double tcount) {
    const double sig1 = sigmoid(g1[t_idx]), sigh = sigmoid(gh[t_idx]);
    const double alpha = sigh / E;
    const double beta = (sig1 - sigh) / tcount;
    const double gamma = -(sig1 - sigh) * P / (tcount * tcount) - sigh / tcount;
    const double zero_order = pr.g0 ? sigmoid(pr.g0[base + t_idx]) / tcount : 0.0;
    unit_vector(q + (size_t)t_idx * d, d, qh.data());
    if (pr.rope) rotate(qh.data(), d, pr.pos0 + t_idx, pr.rope_base);
    double* ot = o + (size_t)t_idx * d;
    for (int j = 0; j < d; ++j) {
      double acc = 0.0;
      for (int a = 0; a < d; ++a) {
        const size_t e = (size_t)a * d + j;
        acc += qh[a] * (alpha * F[e] + beta * G[e] + (gamma + zero_order) * Hs[e]);
      }
      ot[j] = acc;
    }
    if (dbg_s) dbg_s[base + t_idx] = s[t_idx];
    if (dbg_E) dbg_E[base + t_idx] = E;
    if (dbg_P) dbg_P[base + t_idx] = P;
  };

  if (pr.causal) {
    for (int t = 0; t < N; ++t) {
      accumulate(t);
      readout(t, (double)(t + 1));
    }
  } else {
    for (int i = 0; i < N; ++i) accumulate(i);
    for (int t = 0; t < N; ++t) readout(t, (double)N);
  }
}

// Brute-force evaluation of the definition for one (b, h) sequence:
//   softmax_{t,i} = e^{s_i} / E_t, delta_{t,i} = s_i - P_t/t,
//   eps_{t,i} = softmax_{t,i} - 1/t - delta_{t,i}/t,
//   w_{t,i} = sig^1_t delta_{t,i}/t + sig^h_t eps_{t,i}          ([PN] zero-sum weights)
//             (+ sig^0_t / t with the optional zero-order gate)
//   c_{t,i} = q_hat_t R_{t-i} k_hat_i^T                            ([PN] radial-angular + RoPE)
//   o_t = sum_i w_{t,i} c_{t,i} v_i.
// Logits are recomputed from the definition of ubar_i with an explicit inner sum per i.
void brute_one(const Problem& pr, int b, int h, double* out, double* wsum, double* wabsmax) {
  const int N = pr.N, d = pr.d;
  const size_t base = ((size_t)b * pr.H + h) * (size_t)N;
  const double* q = pr.q + base * d;
  const double* k = pr.k + base * d;
  const double* v = pr.v + base * d;
  const double* u = pr.u + base * d;
  const double* mu = pr.mu + (size_t)h * d;
  const double et = std::exp(pr.tau[h]);

  std::vector<double> s(N), ubar(d);
  for (int i = 0; i < N; ++i) {
    const int upto = pr.causal ? i + 1 : N;  // tokens inside the prior mean of token i
    for (int a = 0; a < d; ++a) {
      double acc = 0.0;
      for (int j = 0; j < upto; ++j) acc += u[(size_t)j * d + a];
      ubar[a] = (et * mu[a] + acc) / (et + upto);
    }
    double dot = 0.0;
    for (int a = 0; a < d; ++a) dot += u[(size_t)i * d + a] * ubar[a];
    s[i] = -dot / std::sqrt((double)d);
  }

  std::vector<double> qh(d), kh(d), qr(d);
  for (int t = 0; t < N; ++t) {
    const int last = pr.causal ? t : N - 1;  // tokens i in the weighted sum for query t
    const double tc = (double)(last + 1);
    double E = 0.0, P = 0.0;
    for (int i = 0; i <= last; ++i) {
      E += std::exp(s[i]);
      P += s[i];
    }
    const double sig1 = sigmoid(pr.g1[base + t]), sigh = sigmoid(pr.gh[base + t]);
    const double sig0 = pr.g0 ? sigmoid(pr.g0[base + t]) : 0.0;
    unit_vector(q + (size_t)t * d, d, qh.data());
    double* ot = out + (base + t) * d;
    for (int j = 0; j < d; ++j) ot[j] = 0.0;
    double ws = 0.0, wm = 0.0;
    for (int i = 0; i <= last; ++i) {
      const double soft = std::exp(s[i]) / E;
      const double delta = s[i] - P / tc;
      const double eps = soft - 1.0 / tc - delta / tc;
      const double w_zs = sig1 * delta / tc + sigh * eps;
      const double w = w_zs + sig0 / tc;  // zero-order term (0 unless the gate is given)
      unit_vector(k + (size_t)i * d, d, kh.data());
      std::copy(qh.begin(), qh.end(), qr.begin());
      if (pr.rope) rotate(qr.data(), d, (double)(t - i), pr.rope_base);
      double c = 0.0;
      for (int a = 0; a < d; ++a) c += qr[a] * kh[a];
      const double* vi = v + (size_t)i * d;
      for (int j = 0; j < d; ++j) ot[j] += w * c * vi[j];
      ws += w;
      wm = std::max(wm, std::fabs(w));
    }
    if (wsum) wsum[base + t] = ws;
    if (wabsmax) wabsmax[base + t] = wm;
  }
}

// ZeroS-SM, the quadratic variant: the same zero-sum reweighting applied to standard softmax
// attention ([PN] linear-time prefix scan section: "the same reweighting can be applied to
// standard softmax attention"; the appendix with its formula is not among the pages).  Reading:
// the logits are the standard attention logits s_{t,i} = q_t R_{t-i} k_i^T / sqrt d (raw q and
// k, rotary positions when rope), and every query t has its own softmax, mean logit and
// zero-sum weights over its keys i:
//   softmax_{t,i} = e^{s_{t,i}} / sum_j e^{s_{t,j}},  delta_{t,i} = s_{t,i} - (1/t) sum_j s_{t,j},
//   eps_{t,i} = softmax_{t,i} - 1/t - delta_{t,i}/t,
//   w_{t,i} = sig^1_t delta_{t,i}/t + sig^h_t eps_{t,i} (+ sig^0_t / t),   o_t = sum_i w_{t,i} v_i
// (no angular factor: the logits already carry q and k).  Encoder: every key, t := N.
void sm_one(const Problem& pr, int b, int h, double* out, double* wsum) {
  const int N = pr.N, d = pr.d;
  const size_t base = ((size_t)b * pr.H + h) * (size_t)N;
  const double* q = pr.q + base * d;
  const double* k = pr.k + base * d;
  const double* v = pr.v + base * d;
  std::vector<double> s(N), qr(d);
  for (int t = 0; t < N; ++t) {
    const int last = pr.causal ? t : N - 1;
    const double tc = (double)(last + 1);
    double m = -INFINITY, P = 0.0;
    for (int i = 0; i <= last; ++i) {
      std::copy(q + (size_t)t * d, q + (size_t)(t + 1) * d, qr.begin());
      if (pr.rope) rotate(qr.data(), d, (double)(t - i), pr.rope_base);
      double dot = 0.0;
      for (int a = 0; a < d; ++a) dot += qr[a] * k[(size_t)i * d + a];
      s[i] = dot / std::sqrt((double)d);
      m = std::max(m, s[i]);
      P += s[i];
    }
    double E = 0.0;
    for (int i = 0; i <= last; ++i) E += std::exp(s[i] - m);
    const double sig1 = sigmoid(pr.g1[base + t]), sigh = sigmoid(pr.gh[base + t]);
    const double sig0 = pr.g0 ? sigmoid(pr.g0[base + t]) : 0.0;
    double* ot = out + (base + t) * d;
    for (int j = 0; j < d; ++j) ot[j] = 0.0;
    double ws = 0.0;
    for (int i = 0; i <= last; ++i) {
      const double soft = std::exp(s[i] - m) / E;
      const double delta = s[i] - P / tc;
      const double eps = soft - 1.0 / tc - delta / tc;
      const double w = sig1 * delta / tc + sigh * eps + sig0 / tc;
      for (int j = 0; j < d; ++j) ot[j] += w * v[(size_t)i * d + j];
      ws += w;
    }
    if (wsum) wsum[base + t] = ws;
  }
}

template <class F>
void parallel_over_heads(const Problem& pr, int nthreads, F fn) {
  const int total = pr.B * pr.H;
  if (nthreads <= 0) nthreads = (int)std::max(1u, std::thread::hardware_concurrency());
  nthreads = std::max(1, std::min(nthreads, total));
  std::vector<std::thread> pool;
  for (int w = 0; w < nthreads; ++w)
    pool.emplace_back([&, w] {
      for (int bh = w; bh < total; bh += nthreads) fn(bh / pr.H, bh % pr.H);
    });
  for (auto& th : pool) th.join();
}

bool valid(const Problem& pr) {
  return pr.q && pr.k && pr.v && pr.u && pr.g1 && pr.gh && pr.mu && pr.tau && pr.B >= 0 &&
         pr.H >= 0 && pr.N >= 0 && pr.d > 0 && (pr.d % 2 == 0 || !pr.rope);
}

}  // namespace

extern "C" {

// Recurrent fp64 forward.  Layouts: q,k,v,u,out [B,H,N,d]; g1,gh [B,H,N]; mu [H,d]; tau [H].
// dbg_s/dbg_E/dbg_P ([B,H,N], nullable) receive s_t, E_t and P_t (causal) or s_t, E_N, P_N
// (encoder).  g0 ([B,H,N], nullable) are the zero-order gate logits.  nthreads <= 0 uses every
// hardware thread.  Returns 0, or 1 on bad arguments.
int zs_oracle_fwd(const double* q, const double* k, const double* v, const double* u,
                  const double* g1, const double* gh, const double* mu, const double* tau,
                  double* out, int B, int H, int N, int d, int causal, int rope, double rope_base,
                  double pos0, int nthreads, double* dbg_s, double* dbg_E, double* dbg_P,
                  const double* g0) {
  Problem pr{q, k, v, u, g1, gh, mu, tau, g0, B, H, N, d, causal, rope, rope_base, pos0};
  if (!valid(pr) || !out) return 1;
  parallel_over_heads(pr, nthreads,
                      [&](int b, int h) { recurrent_one(pr, b, h, out, dbg_s, dbg_E, dbg_P); });
  return 0;
}

// Brute-force O(N^2 d) fp64 forward of the definition.  wsum [B,H,N] receives sum_i w_{t,i}
// and wabsmax [B,H,N] receives max_i |w_{t,i}| (both nullable); g0 as in zs_oracle_fwd.
int zs_oracle_brute(const double* q, const double* k, const double* v, const double* u,
                    const double* g1, const double* gh, const double* mu, const double* tau,
                    double* out, int B, int H, int N, int d, int causal, int rope,
                    double rope_base, int nthreads, double* wsum, double* wabsmax,
                    const double* g0) {
  Problem pr{q, k, v, u, g1, gh, mu, tau, g0, B, H, N, d, causal, rope, rope_base, 0.0};
  if (!valid(pr) || !out) return 1;
  parallel_over_heads(pr, nthreads,
                      [&](int b, int h) { brute_one(pr, b, h, out, wsum, wabsmax); });
  return 0;
}

// ZeroS-SM (quadratic variant, see sm_one): q, k, v, out [B,H,N,d]; g1, gh, g0 [B,H,N] (g0
// nullable); wsum [B,H,N] (nullable) receives sum_i w_{t,i}.  Returns 0, or 1 on bad arguments.
int zs_oracle_sm(const double* q, const double* k, const double* v, const double* g1,
                 const double* gh, const double* g0, double* out, int B, int H, int N, int d,
                 int causal, int rope, double rope_base, int nthreads, double* wsum) {
  Problem pr{q, k, v, nullptr, g1, gh, nullptr, nullptr, g0, B, H, N, d, causal, rope,
             rope_base, 0.0};
  if (!q || !k || !v || !g1 || !gh || !out || B < 0 || H < 0 || N < 0 || d <= 0 ||
      (rope && d % 2))
    return 1;
  parallel_over_heads(pr, nthreads, [&](int b, int h) { sm_one(pr, b, h, out, wsum); });
  return 0;
}

// LayerNorm of every output row: o, y [B,H,N,d]; w, b [H,d] (nullable: 1 and 0).  y may alias
// o.  Returns 0, or 1 on bad arguments.
int zs_oracle_layer_norm(const double* o, const double* w, const double* b, double eps, double* y,
                         int B, int H, int N, int d) {
  if (!o || !y || B < 0 || H < 0 || N < 0 || d <= 0 || !(eps >= 0.0)) return 1;
  for (long long r = 0; r < (long long)B * H * N; ++r) {
    const int h = (int)((r / N) % H);
    const double* x = o + r * d;
    double mean = 0.0;
    for (int j = 0; j < d; ++j) mean += x[j];
    mean /= d;
    double var = 0.0;
    for (int j = 0; j < d; ++j) var += (x[j] - mean) * (x[j] - mean);
    var /= d;
    const double inv = 1.0 / std::sqrt(var + eps);
    for (int j = 0; j < d; ++j) {
      const double gain = w ? w[(size_t)h * d + j] : 1.0;
      const double bias = b ? b[(size_t)h * d + j] : 0.0;
      y[r * d + j] = (x[j] - mean) * inv * gain + bias;
    }
  }
  return 0;
}

int zs_oracle_threads(void) { return (int)std::max(1u, std::thread::hardware_concurrency()); }

}  // extern "C"
