// Backward pass of the causal ZeroS layer: gradients of L = sum_t do_t . o_t with respect to
// q, k, v, u, the gate logits g1, gh (and the optional zero-order gate g0), mu and tau.
//
// Method: Paper-Notes "ZeroS: Zero-Sum Linear Attention for Efficient Transformers", method
// details: o_t = q_hat_t W_t with W_t = alpha_t F_t + beta_t G_t + gamma_t H_t (the five-state
// "linear-time prefix scan"), F_t = sum e^{s_i} k_hat_i^T v_i, G_t = sum s_i k_hat_i^T v_i,
// H_t = sum k_hat_i^T v_i, alpha_t = sigh_t/E_t, beta_t = (sig1_t - sigh_t)/t,
// gamma_t = -(sig1_t - sigh_t) P_t/t^2 - sigh_t/t (+ sig0_t/t), and the deviation logits
// s_i = -(1/sqrt d) u_i ubar_i^T with ubar_i = (e^tau mu + sum_{j<=i} u_j)/(e^tau + i).
//
// Differentiating the scan gives, per token:
//   dq_hat_t = do_t W_t^T;  dalpha_t = q_hat_t F_t do_t^T (likewise dbeta_t, dgamma_t with G, H);
//   state gradients D^F_i = sum_{t>=i} alpha_t q_hat_t^T do_t (D^G with beta, D^H with gamma):
//   dk_hat_i = (e^{s_i} D^F_i + s_i D^G_i + D^H_i) v_i^T,
//   dv_i = k_hat_i (e^{s_i} D^F_i + s_i D^G_i + D^H_i),
//   ds_i = e^{s_i} k_hat_i D^F_i v_i^T + k_hat_i D^G_i v_i^T
//          + e^{s_i} sum_{t>=i} dE_t + sum_{t>=i} dP_t,
//     with dE_t = -(sigh_t/E_t^2) dalpha_t and dP_t = -(sig1_t - sigh_t)/t^2 dgamma_t;
//   du_i = -(ds_i ubar_i + Z_i)/sqrt d with Z_i = sum_{j>=i} ds_j u_j/(e^tau + j);
//   dmu = -e^tau Z_1/sqrt d;  dtau = -(e^tau/sqrt d) sum_i ds_i u_i (mu - ubar_i)^T/(e^tau + i);
//   the gates from dalpha, dbeta, dgamma; q and k through the unit normalisation and rotation.
// Everything is kept relative to the running maximum m as in the forward (F~ = F e^{-m},
// Et = E e^{-m}; the suffix sums carry the factor e^{m_i - m_t} <= 1), so no exponential
// overflows.
//
// Structure: one CTA per (b, h) sequence, 256 threads, the d x d matrices in shared memory.
// Pass A runs the tokens in order: the canonical scalar contract of zs_common.cuh (the same s,
// m, Et, P as the forward kernels), the states F~, G, H, and per token dq, the gate gradients
// and the scalars pass B needs (scratch, with ubar_t).  Pass B runs the tokens in reverse with
// the state gradients D~F (= D^F relative to m_i), D^G, D^H and writes dk, dv, du; mu and tau
// gradients are accumulated over the batch with atomics.  A correctness-first CUDA-core kernel
// (O(N d^2) work, like the token-sequential forward).
#include <math.h>

#include <atomic>

#include "zs_common.cuh"
#include "zs_internal.h"

namespace zs {
namespace {

constexpr int kThreads = 256;
constexpr int kScal = 8;  // per-token scalars kept for pass B (followed by ubar_t[d])

template <int D>
struct BwdSmem {
  static constexpr int LD = D + 1;  // padded row stride of the d x d matrices
  static constexpr uint32_t MATS = 3u * D * LD * 4u;
  // 14 vectors of d, the column partials (one per thread) and 64 scalar / reduction slots
  static constexpr uint32_t VECS = (14u * D + kThreads + 64u) * 4u;
  static constexpr uint32_t BYTES = MATS + VECS;
};

// Inverse rotary map of one pair: x = R^T x' (R rotates (a, b) by the angle with (c, s)).
__device__ __forceinline__ void unrotate_pair(float& a, float& b, float2 cs) {
  const float xa = __fmaf_rn(a, cs.x, __fmul_rn(b, cs.y));
  const float xb = __fmaf_rn(-a, cs.y, __fmul_rn(b, cs.x));
  a = xa;
  b = xb;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) bwd_kernel(BwdArgs a) {
  using SM = BwdSmem<D>;
  constexpr int LD = SM::LD;
  constexpr int R = D / 32;          // columns per lane of a warp-owned row (scalar contract)
  constexpr int RS = kThreads / D;   // row groups of the element-wise layout
  constexpr int NR = D / RS;         // matrix rows per thread
  constexpr int TPR = kThreads / D;  // threads per row in the row products
  constexpr int HALF = D / 2;
  extern __shared__ float smf[];
  float* MF = smf;                   // F~ (pass A) / D~F (pass B)
  float* MG = MF + D * LD;           // G / D^G
  float* MH = MG + D * LD;           // H / D^H
  float* vec = MH + D * LD;
  float* qh = vec;                   // rotated unit q_t
  float* qn = qh + D;                // unit q_t (before rotation)
  float* kh = qn + D;
  float* kn = kh + D;
  float* vv = kn + D;
  float* dov = vv + D;               // do_t
  float* yF = dov + D;               // row products
  float* yG = yF + D;
  float* yH = yG + D;
  float* zF = yH + D;                // column products (pass B)
  float* zG = zF + D;
  float* zH = zG + D;
  float* colp = zH + D;              // [RS][D] partial column sums (one per thread)
  float* ub = colp + kThreads;       // ubar_t
  float* uu = ub + D;                // u_t
  float* sc = uu + D;                // small scalars / reduction slots (64)

  const int bh = blockIdx.x, h = bh % a.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = a.N;
  const size_t row0 = (size_t)bh * N;
  const T* __restrict__ q = static_cast<const T*>(a.q) + row0 * D;
  const T* __restrict__ k = static_cast<const T*>(a.k) + row0 * D;
  const T* __restrict__ v = static_cast<const T*>(a.v) + row0 * D;
  const T* __restrict__ u = static_cast<const T*>(a.u) + row0 * D;
  const T* __restrict__ dout = static_cast<const T*>(a.dout) + row0 * D;
  float* scr = a.scratch + row0 * (kScal + D);
  const float etau = expf(a.tau[h]);
  const float rsd = __fdiv_rn(1.0f, __fsqrt_rn((float)D));

  // element-wise layout: thread owns column je = tid % D and rows tid / D + RS r
  const int je = tid % D, re = tid / D;
  // row-product layout: thread handles row ar = tid / TPR, columns jr = pr + TPR i
  const int ar = tid / TPR, pr = tid % TPR;

  for (int e = tid; e < 3 * D * LD; e += kThreads) smf[e] = 0.0f;

  // loads one row: unit vector (before rotation) into un, rotated into ro, and its norm
  auto load_unit = [&](const T* src, int t, float* un, float* ro, float* nrm) {
    // one warp: lane owns columns lane + 32 c
    float x[R];
    float ss = 0.0f;
#pragma unroll
    for (int c = 0; c < R; ++c) {
      x[c] = ld(src, (size_t)t * D + lane + 32 * c);
      ss = __fmaf_rn(x[c], x[c], ss);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    const float n = fmaxf(__fsqrt_rn(ss), 1e-12f);
    const float inv = __fdiv_rn(1.0f, n);
#pragma unroll
    for (int c = 0; c < R; ++c) un[lane + 32 * c] = __fmul_rn(x[c], inv);
    if (lane == 0) *nrm = n;
    __syncwarp();
#pragma unroll
    for (int c = 0; c < R; ++c) {
      const int col = lane + 32 * c;
      float y = un[col];
      if (a.rope) {
        const int pj = col < HALF ? col : col - HALF;
        const float2 cs = a.rope_table[(size_t)t * HALF + pj];
        const float xa = un[pj], xb = un[pj + HALF];
        y = col < HALF ? __fsub_rn(__fmul_rn(xa, cs.x), __fmul_rn(xb, cs.y))
                       : __fadd_rn(__fmul_rn(xa, cs.y), __fmul_rn(xb, cs.x));
      }
      ro[col] = y;
    }
  };

  // gradient through rotation and unit normalisation: dx = (R^T dy - n (n . R^T dy)) / |x|
  // (one warp; dy, un in shared memory; writes fp32 row t of dst)
  auto unit_backward = [&](const float* dy, const float* un, float nrm, int t, float* dst) {
    float g[R];
#pragma unroll
    for (int c = 0; c < R; ++c) {
      const int col = lane + 32 * c;
      float y = dy[col];
      if (a.rope) {
        const int pj = col < HALF ? col : col - HALF;
        const float2 cs = a.rope_table[(size_t)t * HALF + pj];
        float ya = dy[pj], yb = dy[pj + HALF];
        unrotate_pair(ya, yb, cs);
        y = col < HALF ? ya : yb;
      }
      g[c] = y;
    }
    float dot = 0.0f;
#pragma unroll
    for (int c = 0; c < R; ++c) dot = __fmaf_rn(un[lane + 32 * c], g[c], dot);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) dot = __fadd_rn(dot, __shfl_xor_sync(0xffffffffu, dot, o));
    const float inv = __fdiv_rn(1.0f, nrm);
#pragma unroll
    for (int c = 0; c < R; ++c)
      dst[(size_t)t * D + lane + 32 * c] =
          __fmul_rn(__fsub_rn(g[c], __fmul_rn(un[lane + 32 * c], dot)), inv);
  };

  // y[a] = sum_j M[a][j] x[j] for the three matrices at once (TPR threads per row)
  auto row_products = [&](const float* x) {
    float pf = 0.0f, pg = 0.0f, ph = 0.0f;
    for (int j = pr; j < D; j += TPR) {
      const float xj = x[j];
      pf = __fmaf_rn(MF[ar * LD + j], xj, pf);
      pg = __fmaf_rn(MG[ar * LD + j], xj, pg);
      ph = __fmaf_rn(MH[ar * LD + j], xj, ph);
    }
#pragma unroll
    for (int o = TPR / 2; o >= 1; o >>= 1) {
      pf = __fadd_rn(pf, __shfl_xor_sync(0xffffffffu, pf, o));
      pg = __fadd_rn(pg, __shfl_xor_sync(0xffffffffu, pg, o));
      ph = __fadd_rn(ph, __shfl_xor_sync(0xffffffffu, ph, o));
    }
    if (pr == 0) {
      yF[ar] = pf;
      yG[ar] = pg;
      yH[ar] = ph;
    }
  };

  // block sum of one value per thread; every thread gets the result
  auto block_sum = [&](float x, int slot) -> float {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, o));
    if (lane == 0) sc[32 + slot * 8 + warp] = x;
    __syncthreads();
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) s = __fadd_rn(s, sc[32 + slot * 8 + w]);
    __syncthreads();
    return s;
  };

  // ================================================================ pass A (token order)
  float C[R], L[R], mu[R];
  Scalars scs = scalars_init();
  if (warp == 0) {
#pragma unroll
    for (int c = 0; c < R; ++c) {
      C[c] = 0.0f;
      L[c] = 0.0f;
      mu[c] = a.mu[(size_t)h * D + R * lane + c];
    }
  }
  __syncthreads();
  for (int t = 0; t < N; ++t) {
    if (warp == 0) {
      float ux[R];
#pragma unroll
      for (int c = 0; c < R; ++c) ux[c] = ld(u, (size_t)t * D + R * lane + c);
      const TokenOut o = token_update<R>(ux, C, L, mu, etau, t + 1, scs);
      // ubar_t = (e^tau mu + S_t) / (e^tau + t) with S_t = C + L after the update
      const float dent = __fdiv_rn(1.0f, __fadd_rn(etau, (float)(t + 1)));
#pragma unroll
      for (int c = 0; c < R; ++c)
        scr[(size_t)t * (kScal + D) + kScal + R * lane + c] =
            __fmul_rn(__fmaf_rn(etau, mu[c], __fadd_rn(C[c], L[c])), dent);
      if (lane == 0) {
        if (!isfinite(o.s)) report(a.status, kErrRange);
        const float sig1 = sigmoid(a.g1[row0 + t]), sigh = sigmoid(a.gh[row0 + t]);
        const float rt = __fdiv_rn(1.0f, (float)(t + 1));
        const float beta = __fmul_rn(__fsub_rn(sig1, sigh), rt);
        float gamma = -__fadd_rn(__fmul_rn(__fmul_rn(beta, o.P), rt), __fmul_rn(sigh, rt));
        if (a.g0) gamma = __fadd_rn(gamma, __fmul_rn(sigmoid(a.g0[row0 + t]), rt));
        sc[0] = o.s;
        sc[1] = o.m;
        sc[2] = o.Et;
        sc[3] = __fdiv_rn(sigh, o.Et);  // alpha~ = alpha e^{m}
        sc[4] = beta;
        sc[5] = gamma;
        sc[6] = expf(__fsub_rn(o.m_prev, o.m));  // rescale of F~
        sc[7] = expf(__fsub_rn(o.s, o.m));       // e^{s - m}
        sc[8] = o.P;
        sc[9] = sig1;
        sc[10] = sigh;
      }
    } else if (warp == 1) {
      load_unit(q, t, qn, qh, &sc[16]);
    } else if (warp == 2) {
      load_unit(k, t, kn, kh, &sc[17]);
    } else if (warp == 3) {
#pragma unroll
      for (int c = 0; c < R; ++c) {
        vv[lane + 32 * c] = ld(v, (size_t)t * D + lane + 32 * c);
        dov[lane + 32 * c] = ld(dout, (size_t)t * D + lane + 32 * c);
      }
    }
    __syncthreads();
    {  // states after token t
      const float f = sc[6], g = sc[7], s = sc[0];
      const float vj = vv[je];
#pragma unroll 4
      for (int r = 0; r < NR; ++r) {
        const int ai = re + RS * r;
        const float kv = __fmul_rn(kh[ai], vj);
        MF[ai * LD + je] = __fmaf_rn(MF[ai * LD + je], f, __fmul_rn(g, kv));
        MG[ai * LD + je] = __fmaf_rn(s, kv, MG[ai * LD + je]);
        MH[ai * LD + je] = __fadd_rn(MH[ai * LD + je], kv);
      }
    }
    __syncthreads();
    row_products(dov);
    __syncthreads();
    // dq_hat = alpha~ F~ do + beta G do + gamma H do; dalpha~, dbeta, dgamma = q_hat . (.)
    float pa = 0.0f, pb = 0.0f, pgm = 0.0f;
    if (tid < D) {
      const float dqh = __fmaf_rn(sc[3], yF[tid], __fmaf_rn(sc[4], yG[tid], __fmul_rn(sc[5], yH[tid])));
      zF[tid] = dqh;  // dq_hat staged for the normalisation backward
      pa = __fmul_rn(qh[tid], yF[tid]);
      pb = __fmul_rn(qh[tid], yG[tid]);
      pgm = __fmul_rn(qh[tid], yH[tid]);
    }
    const float dal = block_sum(pa, 0);
    const float dbe = block_sum(pb, 1);
    const float dga = block_sum(pgm, 2);
    if (warp == 1) unit_backward(zF, qn, sc[16], t, a.dq + row0 * D);
    if (tid == 0) {
      const float tf = (float)(t + 1);
      const float rt = __fdiv_rn(1.0f, tf);
      const float P = sc[8], sig1 = sc[9], sigh = sc[10];
      const float Pt2 = __fmul_rn(__fmul_rn(P, rt), rt);
      const float dsig1 = __fsub_rn(__fmul_rn(dbe, rt), __fmul_rn(dga, Pt2));
      const float dsigh = __fadd_rn(__fsub_rn(__fdiv_rn(dal, sc[2]), __fmul_rn(dbe, rt)),
                                    __fmul_rn(dga, __fsub_rn(Pt2, rt)));
      a.dg1[row0 + t] = __fmul_rn(dsig1, __fmul_rn(sig1, __fsub_rn(1.0f, sig1)));
      a.dgh[row0 + t] = __fmul_rn(dsigh, __fmul_rn(sigh, __fsub_rn(1.0f, sigh)));
      if (a.g0 && a.dg0) {
        const float s0 = sigmoid(a.g0[row0 + t]);
        a.dg0[row0 + t] = __fmul_rn(__fmul_rn(dga, rt), __fmul_rn(s0, __fsub_rn(1.0f, s0)));
      }
      float* rs = scr + (size_t)t * (kScal + D);
      rs[0] = sc[0];  // s
      rs[1] = sc[1];  // m
      rs[2] = sc[2];  // Et
      rs[3] = sc[3];  // alpha~
      rs[4] = sc[4];  // beta
      rs[5] = sc[5];  // gamma
      rs[6] = dal;    // dalpha~
      rs[7] = dga;    // dgamma
    }
    __syncthreads();
  }

  // ================================================================ pass B (reverse order)
  for (int e = tid; e < 3 * D * LD; e += kThreads) smf[e] = 0.0f;
  float zacc = 0.0f, tacc = 0.0f;  // thread a < D: Z[a] and its dtau partial
  float EA = 0.0f, PA = 0.0f;  // thread 0: suffix sums of dE e^{m} and dP
  float m_next = 0.0f;         // m_{t+1}
  const float mu_a = tid < D ? a.mu[(size_t)h * D + tid] : 0.0f;
  __syncthreads();
  for (int t = N - 1; t >= 0; --t) {
    const float* rs = scr + (size_t)t * (kScal + D);
    if (warp == 0) {
      if (lane < kScal) sc[lane] = rs[lane];
#pragma unroll
      for (int c = 0; c < R; ++c) {
        ub[lane + 32 * c] = rs[kScal + lane + 32 * c];
        uu[lane + 32 * c] = ld(u, (size_t)t * D + lane + 32 * c);
      }
    } else if (warp == 1) {
      load_unit(q, t, qn, qh, &sc[16]);
    } else if (warp == 2) {
      load_unit(k, t, kn, kh, &sc[17]);
    } else if (warp == 3) {
#pragma unroll
      for (int c = 0; c < R; ++c) {
        vv[lane + 32 * c] = ld(v, (size_t)t * D + lane + 32 * c);
        dov[lane + 32 * c] = ld(dout, (size_t)t * D + lane + 32 * c);
      }
    }
    __syncthreads();
    const float s = sc[0], m = sc[1], Et = sc[2], alt = sc[3], beta = sc[4], gamma = sc[5];
    const float dal = sc[6], dga = sc[7];
    const float resc = (t == N - 1) ? 0.0f : expf(__fsub_rn(m, m_next));  // e^{m_t - m_{t+1}}
    {  // D~F = e^{m_t - m_{t+1}} D~F + alpha~ q_hat^T do, D^G += beta q_hat^T do, D^H += ...
      const float dj = dov[je];
#pragma unroll 4
      for (int r = 0; r < NR; ++r) {
        const int ai = re + RS * r;
        const float qd = __fmul_rn(qh[ai], dj);
        MF[ai * LD + je] = __fmaf_rn(MF[ai * LD + je], resc, __fmul_rn(alt, qd));
        MG[ai * LD + je] = __fmaf_rn(beta, qd, MG[ai * LD + je]);
        MH[ai * LD + je] = __fmaf_rn(gamma, qd, MH[ai * LD + je]);
      }
    }
    __syncthreads();
    row_products(vv);  // yF = D~F v, yG = D^G v, yH = D^H v
    {                  // column products k_hat D: partial sums over this thread's rows
      float cf = 0.0f, cg = 0.0f, chh = 0.0f;
#pragma unroll 4
      for (int r = 0; r < NR; ++r) {
        const int ai = re + RS * r;
        const float kk = kh[ai];
        cf = __fmaf_rn(kk, MF[ai * LD + je], cf);
        cg = __fmaf_rn(kk, MG[ai * LD + je], cg);
        chh = __fmaf_rn(kk, MH[ai * LD + je], chh);
      }
      // RS partials per column: combine through shared memory (3 passes of the same buffer)
      colp[re * D + je] = cf;
      __syncthreads();
      if (tid < D) {
        float x = 0.0f;
        for (int g = 0; g < RS; ++g) x = __fadd_rn(x, colp[g * D + tid]);
        zF[tid] = x;
      }
      __syncthreads();
      colp[re * D + je] = cg;
      __syncthreads();
      if (tid < D) {
        float x = 0.0f;
        for (int g = 0; g < RS; ++g) x = __fadd_rn(x, colp[g * D + tid]);
        zG[tid] = x;
      }
      __syncthreads();
      colp[re * D + je] = chh;
      __syncthreads();
      if (tid < D) {
        float x = 0.0f;
        for (int g = 0; g < RS; ++g) x = __fadd_rn(x, colp[g * D + tid]);
        zH[tid] = x;
      }
      __syncthreads();
    }
    const float ex = expf(__fsub_rn(s, m));  // e^{s_t - m_t}
    float pk = 0.0f, pg2 = 0.0f;
    if (tid < D) {
      // dk_hat and dv of this token; dk_hat staged in yG's slot after use
      const float dkh = __fmaf_rn(ex, yF[tid], __fmaf_rn(s, yG[tid], yH[tid]));
      const float dvv = __fmaf_rn(ex, zF[tid], __fmaf_rn(s, zG[tid], zH[tid]));
      a.dv[(row0 + t) * D + tid] = dvv;
      pk = __fmul_rn(kh[tid], yF[tid]);
      pg2 = __fmul_rn(kh[tid], yG[tid]);
      zH[tid] = dkh;
    }
    const float kf = block_sum(pk, 0);
    const float kg = block_sum(pg2, 1);
    if (tid == 0) {
      const float tf = (float)(t + 1);
      EA = __fmaf_rn(EA, resc, -__fdiv_rn(__fmul_rn(alt, dal), Et));
      PA = __fsub_rn(PA, __fmul_rn(__fdiv_rn(beta, tf), dga));
      const float ds = __fadd_rn(__fmaf_rn(ex, kf, kg), __fmaf_rn(ex, EA, PA));
      sc[12] = ds;
    }
    m_next = m;  // every thread rescales the state gradients with e^{m_t - m_{t+1}}
    if (warp == 2) unit_backward(zH, kn, sc[17], t, a.dk + row0 * D);
    __syncthreads();
    const float ds = sc[12];
    if (tid < D) {
      const float w = __fdiv_rn(1.0f, __fadd_rn(etau, (float)(t + 1)));
      const float ua = uu[tid], uba = ub[tid];
      zacc = __fmaf_rn(__fmul_rn(ds, ua), w, zacc);
      tacc = __fmaf_rn(__fmul_rn(__fmul_rn(ds, ua), __fsub_rn(mu_a, uba)), w, tacc);
      a.du[(row0 + t) * D + tid] = -__fmul_rn(__fmaf_rn(ds, uba, zacc), rsd);
    }
    __syncthreads();
  }
  // mu and tau: summed over the batch (atomics; the host zeroes them first)
  const float tsum = block_sum(tid < D ? tacc : 0.0f, 2);
  if (tid < D) atomicAdd(a.dmu + (size_t)h * D + tid, -__fmul_rn(__fmul_rn(etau, zacc), rsd));
  if (tid == 0) atomicAdd(a.dtau + h, -__fmul_rn(__fmul_rn(etau, tsum), rsd));
}

template <typename T, int D>
cudaError_t launch_t(const BwdArgs& a, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(bwd_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)BwdSmem<D>::BYTES);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  bwd_kernel<T, D><<<a.B * a.H, kThreads, BwdSmem<D>::BYTES, stream>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_scratch_bytes(int B, int H, int N, int d) {
  return (size_t)B * H * N * (kScal + d) * sizeof(float);
}

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream) {
  const bool f32 = a.dtype == 1;
  switch (a.d) {
    case 32: return f32 ? launch_t<float, 32>(a, stream) : launch_t<__nv_bfloat16, 32>(a, stream);
    case 64: return f32 ? launch_t<float, 64>(a, stream) : launch_t<__nv_bfloat16, 64>(a, stream);
    case 128:
      return f32 ? launch_t<float, 128>(a, stream) : launch_t<__nv_bfloat16, 128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace zs
