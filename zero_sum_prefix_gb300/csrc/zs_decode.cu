// Recurrent-inference step of the ZeroS layer: one new token for every (b, h) sequence.
//
// Method: Paper-Notes "ZeroS: Zero-Sum Linear Attention for Efficient Transformers", method
// details, "linear-time prefix scan" (O(d^2) state, O(d^2) work per step): the token updates
// E, P, F, G, H and is read out as o_t = q_hat_t (alpha_t F_t + beta_t G_t + gamma_t H_t).
// The scalars follow the canonical token update of zs_common.cuh, so s, P, m and Et are
// bit-identical to those of the forward kernels for the same token.
//
// The step is bound by HBM bandwidth: it streams the three fp32 d x d matrices of every
// sequence in and out (24 d^2 bytes) and touches O(d) bytes of token data.  One CTA per
// (b, h); 256 threads; thread (rp, c4) updates float4 column group c4 of rows rp, rp + RPP, ...
// of F~, G and H in one pass (load, rank-1 update, readout partial, store), so each state byte
// is read once and written once.
#include <math.h>

#include "zs_common.cuh"
#include "zs_internal.h"

namespace zs {
namespace {

constexpr int kThreads = 256;

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) decode_kernel(DecodeArgs a) {
  constexpr int R = D / 32;
  constexpr int C4 = D / 4;             // float4 per state row
  constexpr int RPP = kThreads / C4;    // rows per pass
  constexpr int PASSES = D / RPP;
  constexpr int UNR = PASSES < 4 ? PASSES : 4;
  const int bh = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* rec = record_ptr(a.state, bh, D);
  RecordHead* hd = reinterpret_cast<RecordHead*>(rec);

  __shared__ float qs[D], ks[D], vs[D];
  __shared__ float coef[6];  // s, f, g, alpha, beta, gamma
  __shared__ float4 red[RPP][C4];

  const int t_old = hd->t;
  const size_t tok = (size_t)bh * D;
  const T* __restrict__ q = static_cast<const T*>(a.q) + tok;
  const T* __restrict__ k = static_cast<const T*>(a.k) + tok;
  const T* __restrict__ v = static_cast<const T*>(a.v) + tok;
  const T* __restrict__ u = static_cast<const T*>(a.u) + tok;

  float C[R], L[R];
  Scalars sc;
  if (warp == 0) {
    float uu[R], mu[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      uu[r] = ld(u, R * lane + r);
      C[r] = rec[rec_C(D) + R * lane + r];
      L[r] = rec[rec_L(D) + R * lane + r];
      mu[r] = rec[rec_mu(D) + R * lane + r];
    }
    sc.mC = hd->mC;
    sc.EC = hd->EC;
    sc.CP = hd->CP;
    sc.ml = hd->ml;
    sc.El = hd->El;
    sc.LP = hd->LP;
    const float etau = hd->etau;
    const TokenOut o = token_update<R>(uu, C, L, mu, etau, t_old + 1, sc);
    const float s = o.s;
    const float f = expf(__fsub_rn(o.m_prev, o.m));
    const float g = expf(__fsub_rn(s, o.m));
    if (lane == 0) {
      if (!isfinite(s)) report(a.status, kErrRange);
      const float sig1 = sigmoid(a.g1[bh]), sigh = sigmoid(a.gh[bh]);
      const float rt = __fdiv_rn(1.0f, (float)(t_old + 1));
      const float beta = __fmul_rn(__fsub_rn(sig1, sigh), rt);
      coef[0] = s;
      coef[1] = f;
      coef[2] = g;
      coef[3] = __fdiv_rn(sigh, o.Et);
      coef[4] = beta;
      coef[5] = -__fadd_rn(__fmul_rn(__fmul_rn(beta, o.P), rt), __fmul_rn(sigh, rt));
      // optional zero-order term of a first layer: every weight gains sig0 / t
      if (a.g0) coef[5] = __fadd_rn(coef[5], __fmul_rn(sigmoid(a.g0[bh]), rt));
      if (a.dbg_s) a.dbg_s[bh] = s;
      if (a.dbg_E) a.dbg_E[bh] = o.Et;
      if (a.dbg_P) a.dbg_P[bh] = o.P;
      if (a.dbg_m) a.dbg_m[bh] = o.m;
    }
  } else if (warp == 1 || warp == 2) {
    const T* src = warp == 1 ? q : k;
    float x[R];
    float2 cs[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      x[r] = ld(src, lane + 32 * r);
      cs[r] = make_float2(1.0f, 0.0f);
    }
    if (a.rope) {
      if (R == 1) {
        cs[0] = rope_cs((double)t_old, pair_index<R>(lane, 0), D, (double)a.rope_base);
      } else {
#pragma unroll
        for (int r = 0; r < R / 2; ++r)
          cs[r] = rope_cs((double)t_old, pair_index<R>(lane, r), D, (double)a.rope_base);
      }
    }
    unit_rotate<R>(x, a.rope != 0, cs);
    float* dst = warp == 1 ? qs : ks;
#pragma unroll
    for (int r = 0; r < R; ++r) dst[lane + 32 * r] = x[r];
  } else if (warp == 3) {
#pragma unroll
    for (int r = 0; r < R; ++r) vs[lane + 32 * r] = ld(v, lane + 32 * r);
  }
  __syncthreads();

  const float s = coef[0], f = coef[1], g = coef[2];
  const float alpha = coef[3], beta = coef[4], gamma = coef[5];
  const int c4 = threadIdx.x % C4, rp = threadIdx.x / C4;
  const float4 v4 = reinterpret_cast<const float4*>(vs)[c4];
  float4* Fp = reinterpret_cast<float4*>(rec + rec_F(D)) + c4;
  float4* Gp = reinterpret_cast<float4*>(rec + rec_G(D)) + c4;
  float4* Hp = reinterpret_cast<float4*>(rec + rec_H(D)) + c4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);

  for (int p0 = 0; p0 < PASSES; p0 += UNR) {
    float4 Fv[UNR], Gv[UNR], Hv[UNR];
#pragma unroll
    for (int i = 0; i < UNR; ++i) {
      const int row = (p0 + i) * RPP + rp;
      Fv[i] = Fp[row * C4];
      Gv[i] = Gp[row * C4];
      Hv[i] = Hp[row * C4];
    }
#pragma unroll
    for (int i = 0; i < UNR; ++i) {
      const int row = (p0 + i) * RPP + rp;
      const float kr = ks[row], qr = qs[row];
      float* fv = reinterpret_cast<float*>(&Fv[i]);
      float* gv = reinterpret_cast<float*>(&Gv[i]);
      float* hv = reinterpret_cast<float*>(&Hv[i]);
      const float* vv = reinterpret_cast<const float*>(&v4);
      float* ac = reinterpret_cast<float*>(&acc);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float kv = __fmul_rn(kr, vv[c]);
        fv[c] = __fmaf_rn(fv[c], f, __fmul_rn(g, kv));
        gv[c] = __fmaf_rn(s, kv, gv[c]);
        hv[c] = __fadd_rn(hv[c], kv);
        const float comb = __fmaf_rn(alpha, fv[c], __fmaf_rn(beta, gv[c], __fmul_rn(gamma, hv[c])));
        ac[c] = __fmaf_rn(qr, comb, ac[c]);
      }
      Fp[row * C4] = Fv[i];
      Gp[row * C4] = Gv[i];
      Hp[row * C4] = Hv[i];
    }
  }
  red[rp][c4] = acc;
  __syncthreads();
  if (warp == 0) {  // lanes < C4 reduce and write 4 output columns each
    const bool mine = threadIdx.x < C4;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (mine) {
      o = red[0][threadIdx.x];
#pragma unroll 4
      for (int r = 1; r < RPP; ++r) {
        const float4 x = red[r][threadIdx.x];
        o.x = __fadd_rn(o.x, x.x);
        o.y = __fadd_rn(o.y, x.y);
        o.z = __fadd_rn(o.z, x.z);
        o.w = __fadd_rn(o.w, x.w);
      }
    }
    if (a.ln) {  // output LayerNorm over the head's d columns (mean first, then deviations)
      const float mean = warp_sum32((o.x + o.y) + (o.z + o.w)) * (1.0f / D);
      float dv = 0.0f;
      if (mine)
        dv = (o.x - mean) * (o.x - mean) + (o.y - mean) * (o.y - mean) +
             (o.z - mean) * (o.z - mean) + (o.w - mean) * (o.w - mean);
      const float rstd = rsqrtf(warp_sum32(dv) * (1.0f / D) + a.ln_eps);
      if (mine) {
        // gain and bias rows are 16-byte aligned (checked by the host)
        const size_t j4 = ((size_t)(bh % a.H) * D) / 4 + threadIdx.x;
        const float4 w = a.ln_w ? reinterpret_cast<const float4*>(a.ln_w)[j4]
                                : make_float4(1.f, 1.f, 1.f, 1.f);
        const float4 b = a.ln_b ? reinterpret_cast<const float4*>(a.ln_b)[j4]
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        o.x = __fmaf_rn((o.x - mean) * rstd, w.x, b.x);
        o.y = __fmaf_rn((o.y - mean) * rstd, w.y, b.y);
        o.z = __fmaf_rn((o.z - mean) * rstd, w.z, b.z);
        o.w = __fmaf_rn((o.w - mean) * rstd, w.w, b.w);
      }
    }
    if (mine) {
      T* out = static_cast<T*>(a.out) + tok + 4 * threadIdx.x;
      st(out, 0, o.x);
      st(out, 1, o.y);
      st(out, 2, o.z);
      st(out, 3, o.w);
    }
  }
  if (warp == 0) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      rec[rec_C(D) + R * lane + r] = C[r];
      rec[rec_L(D) + R * lane + r] = L[r];
    }
    if (lane == 0) {
      hd->t = t_old + 1;
      hd->mC = sc.mC;
      hd->EC = sc.EC;
      hd->CP = sc.CP;
      hd->ml = sc.ml;
      hd->El = sc.El;
      hd->LP = sc.LP;
    }
  }
}

template <typename T>
cudaError_t launch_typed(const DecodeArgs& a, cudaStream_t stream) {
  const int grid = a.B * a.H;
  switch (a.d) {
    case 32: decode_kernel<T, 32><<<grid, kThreads, 0, stream>>>(a); break;
    case 64: decode_kernel<T, 64><<<grid, kThreads, 0, stream>>>(a); break;
    case 128: decode_kernel<T, 128><<<grid, kThreads, 0, stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.B * a.H == 0) return cudaSuccess;
  return a.dtype == 1 ? launch_typed<float>(a, stream) : launch_typed<__nv_bfloat16>(a, stream);
}

}  // namespace zs
