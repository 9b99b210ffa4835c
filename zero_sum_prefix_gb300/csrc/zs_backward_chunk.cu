// Chunk-parallel backward of the causal ZeroS layer (d = 64): the same gradients as the
// token-sequential kernel of zs_backward.cu (Paper-Notes "ZeroS: Zero-Sum Linear Attention for
// Efficient Transformers", method details: deviation logits, zero-sum weights, radial-angular
// decoupling, linear-time prefix scan; the derivative of that definition), computed in chunks
// of C = 64 tokens so that every (b, h, chunk) works in parallel.
//
// With W_{t,i} = alpha_t e^{s_i} + beta_t s_i + gamma_t and c_{t,i} = q_hat_t k_hat_i^T, the
// output is o_t = sum_{i<=t} c_{t,i} W_{t,i} v_i.  For a chunk c (reference M_c = running max at
// its last token, M_{c-1} at the previous chunk's), in fp32:
//   intra:  S = Q K^T, dA = dO V^T, W~_{t,i} = ah_t e_i + beta_t s_i + gamma_t (i <= t, inside the
//           chunk; e_i = e^{s_i - M_c}, ah_t = alpha~_t e^{M_c - m_t}), A = S o W~, dC = dA o W~,
//           dW = dA o S;  dQ += dC K, dK += dC^T Q, dV += A^T dO;  row sums of dW (e, s, 1)
//           give the intra parts of d ah, d beta, d gamma; column sums (ah, beta) the direct ds.
//   inter (the chunk-start states F~_c = sum_{i<chunk} e^{s_i - M_{c-1}} k_i^T v_i, G_c, H_c):
//           X = dO [F~|G|H]^T; dq_hat += rho X_F + beta X_G + gamma X_H (rho_t = alpha~_t
//           e^{M_{c-1} - m_t}); d rho, d beta, d gamma += q_hat . X.
//   suffix (the states of the later chunks D~F_c = sum_{t>chunk} alpha~_t e^{M_c - m_t} q^T do,
//           D^G_c, D^H_c): Y = V D^T, Z = K D;  dk_hat += e Y_F + s Y_G + Y_H,
//           dv += e Z_F + s Z_G + Z_H, ds += e v.Z_F + v.Z_G.
// The chunk-start and suffix states come from bwd_states_kernel (one pass over the chunks in
// each direction, all value columns in one CTA); the E and P terms of ds, the gate
// gradients' companions and du, d mu, d tau from bwd_ds_kernel and bwd_du_kernel (scans over
// the tokens).
// The per-token s, E e^{-m}, P and m are those of the forward kernels (their debug outputs).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include <atomic>

#include "zs_common.cuh"
#include "zs_internal.h"
#include "zs_tiles.cuh"

namespace zs {
namespace {

using tiles::gemm64;
using tiles::sum16;
using tiles::zero44;

constexpr int kD = 64;        // head dimension of the chunked path
constexpr int kCk = 64;       // tokens per chunk
constexpr int kNT = 256;      // threads per CTA
constexpr int kLD = tiles::kLD;  // padded row stride of the fp32 tiles

// Scratch layout (fp32), shared with the host: per-token forward scalars, the two state sets,
// per-token backward scalars, the prior means.
struct BwdChunkScratch {
  float *s, *E, *P, *m;   // [BH][N] forward scalars (s, E e^{-m}, P, m)
  float* fs;              // [BH][NC][3][D][D] chunk-start states F~, G, H
  float* ds;              // [BH][NC][3][D][D] suffix states D~F, D^G, D^H
  float* tok;             // [BH][N][4] d alpha~, d gamma, direct ds, ds
  float* ubar;            // [BH][N][D]
  float *qhat, *khat;     // [BH][N][D] rotated unit q and k
  float *nq, *nk;         // [BH][N] their norms
};

// Token coefficients of the forward (the same expressions as the forward kernels).
struct TokCoef {
  float alt, beta, gamma, sig1, sigh;
};
__device__ __forceinline__ TokCoef tok_coef(const BwdArgs& a, size_t row, int t, float Et,
                                            float P) {
  TokCoef c;
  c.sig1 = sigmoid(a.g1[row]);
  c.sigh = sigmoid(a.gh[row]);
  const float rt = __fdiv_rn(1.0f, (float)(t + 1));
  c.beta = __fmul_rn(__fsub_rn(c.sig1, c.sigh), rt);
  c.gamma = -__fadd_rn(__fmul_rn(__fmul_rn(c.beta, P), rt), __fmul_rn(c.sigh, rt));
  if (a.g0) c.gamma = __fadd_rn(c.gamma, __fmul_rn(sigmoid(a.g0[row]), rt));
  c.alt = __fdiv_rn(c.sigh, Et);
  return c;
}

// Rotated unit vector of row t of src (one warp; lane owns columns lane and lane + 32, which
// form one rotary pair).  Returns the norm; writes the rotated unit row to dst[0..64).
template <typename T>
__device__ __forceinline__ float unit_row(const T* src, const BwdArgs& a, int t, float* dst) {
  const int lane = threadIdx.x & 31;
  float x0 = ld(src, lane), x1 = ld(src, lane + 32);
  float ss = __fmaf_rn(x0, x0, __fmul_rn(x1, x1));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
  const float n = fmaxf(__fsqrt_rn(ss), 1e-12f);
  const float inv = __fdiv_rn(1.0f, n);
  x0 = __fmul_rn(x0, inv);
  x1 = __fmul_rn(x1, inv);
  if (a.rope) {
    const float2 cs = a.rope_table[(size_t)t * (kD / 2) + lane];
    const float y0 = __fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, cs.y));
    const float y1 = __fadd_rn(__fmul_rn(x0, cs.y), __fmul_rn(x1, cs.x));
    x0 = y0;
    x1 = y1;
  }
  dst[lane] = x0;
  dst[lane + 32] = x1;
  return n;
}

// ================================================================== unit rows
// Rotated unit vectors of every q and k row (one warp per row), with the norms.
template <typename T>
__global__ void __launch_bounds__(kNT) bwd_rows_kernel(BwdArgs a, BwdChunkScratch sc) {
  const size_t rows = (size_t)a.B * a.H * a.N;
  const int lane = threadIdx.x & 31;
  for (size_t w = (blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5; w < 2 * rows;
       w += ((size_t)gridDim.x * blockDim.x) >> 5) {
    const bool isk = w >= rows;
    const size_t row = isk ? w - rows : w;
    const int t = (int)(row % a.N);
    const T* src = static_cast<const T*>(isk ? a.k : a.q) + row * kD;
    const float n = unit_row<T>(src, a, t, (isk ? sc.khat : sc.qhat) + row * kD);
    if (lane == 0) (isk ? sc.nk : sc.nq)[row] = n;
  }
}

// ================================================================== chunk states
// grid (BH, 1, 2): z = 0 stores the chunk-start forward states F~_c, G_c, H_c (F~ relative to
// M_{c-1}) going forward; z = 1 stores the suffix states D~F_c (relative to M_c), D^G_c, D^H_c
// going backward.  Thread (ar = tid / 16, cj = tid % 16) holds rows 4 ar .. 4 ar + 3 and columns
// 4 cj .. 4 cj + 3 of each d x d state (48 accumulators: per token 16 products and 48
// multiply-adds against three 16-byte shared-memory loads).  The next chunk's rows, values and
// scalars are loaded into registers while the current chunk is accumulated.
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  float4 r;
  r.x = __uint_as_float(w.x << 16);
  r.y = __uint_as_float(w.x & 0xffff0000u);
  r.z = __uint_as_float(w.y << 16);
  r.w = __uint_as_float(w.y & 0xffff0000u);
  return r;
}

template <typename T>
__global__ void __launch_bounds__(kNT) bwd_states_kernel(BwdArgs a, BwdChunkScratch sc) {
  __shared__ __align__(16) float rows[kCk][kD];  // k_hat (z = 0) or q_hat (z = 1) of the chunk
  __shared__ __align__(16) float cols[kCk][kD];  // v or do of the chunk
  __shared__ __align__(16) float cf[kCk][4];     // per-token weights of the three states
  __shared__ float fac;                          // rescale of the F~ state
  const int bh = blockIdx.x, dir = blockIdx.z;
  const int N = a.N, NC = (N + kCk - 1) / kCk;
  const int tid = threadIdx.x;
  const int ar = tid >> 4, cj = tid & 15;
  const size_t row0 = (size_t)bh * N;
  const float* __restrict__ hat = (dir == 0 ? sc.khat : sc.qhat) + row0 * kD;
  const T* __restrict__ val = static_cast<const T*>(dir == 0 ? a.v : a.dout) + row0 * kD;
  float st[3][4][4];
#pragma unroll
  for (int m = 0; m < 3; ++m)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) st[m][i][j] = 0.0f;
  float* out = dir == 0 ? sc.fs : sc.ds;
  // prefetch registers: 16 row values, 16 values, the token's weights, M_c, M_{c-1}
  float4 pr[4], pv[4];
  float pw[3], pMc = 0.0f, pMp = 0.0f;
  auto fetch = [&](int c) {
    const int t0 = c * kCk, tn = min(N, t0 + kCk) - t0;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int e = tid + kNT * x, r = e / (kD / 4);
      const float4 z = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      pr[x] = r < tn ? reinterpret_cast<const float4*>(hat + (size_t)t0 * kD)[e] : z;
      pv[x] = r < tn ? ld4(val + (size_t)t0 * kD + 4 * (size_t)e) : z;
    }
    pMc = sc.m[row0 + t0 + tn - 1];
    pMp = c > 0 ? sc.m[row0 + t0 - 1] : 0.0f;
    pw[0] = pw[1] = pw[2] = 0.0f;
    if (tid < tn) {
      const size_t row = row0 + t0 + tid;
      const float s = sc.s[row];
      if (dir == 0) {
        pw[0] = expf(__fsub_rn(s, pMc));  // e_i relative to M_c
        pw[1] = s;
        pw[2] = 1.0f;
      } else {
        const TokCoef k = tok_coef(a, row, t0 + tid, sc.E[row], sc.P[row]);
        pw[0] = __fmul_rn(k.alt, expf(__fsub_rn(pMp, sc.m[row])));  // relative to M_{c-1}
        pw[1] = k.beta;
        pw[2] = k.gamma;
      }
    }
  };
  const int last = dir == 0 ? NC - 1 : 0;  // the chunk whose state is stored without an update
  if (NC > 1) fetch(dir == 0 ? 0 : NC - 1);
  for (int it = 0; it < NC; ++it) {
    const int c = dir == 0 ? it : NC - 1 - it;
    float* dst = out + (((size_t)bh * NC + c) * 3) * kD * kD;
#pragma unroll
    for (int m = 0; m < 3; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4*>(dst + (size_t)m * kD * kD + (4 * ar + i) * kD + 4 * cj) =
            make_float4(st[m][i][0], st[m][i][1], st[m][i][2], st[m][i][3]);
    if (c == last) break;
    const int tn = min(N, c * kCk + kCk) - c * kCk;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      reinterpret_cast<float4*>(&rows[0][0])[tid + kNT * x] = pr[x];
      reinterpret_cast<float4*>(&cols[0][0])[tid + kNT * x] = pv[x];
    }
    if (tid < kCk) *reinterpret_cast<float4*>(&cf[tid][0]) = make_float4(pw[0], pw[1], pw[2], 0.0f);
    if (tid == 0) fac = (dir == 0 && c == 0) ? 0.0f : expf(__fsub_rn(pMp, pMc));
    __syncthreads();
    const int nxt = dir == 0 ? c + 1 : c - 1;
    if (nxt != last) fetch(nxt);  // in flight while this chunk is accumulated
    const float f = fac;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) st[0][i][j] = __fmul_rn(st[0][i][j], f);
#pragma unroll 2
    for (int r = 0; r < tn; ++r) {
      // packed fp32 pairs (columns j, j + 1): the same roundings as scalar products and fmas
      const float4 k4 = *reinterpret_cast<const float4*>(&rows[r][4 * ar]);
      const float4 v4 = *reinterpret_cast<const float4*>(&cols[r][4 * cj]);
      const float4 w = *reinterpret_cast<const float4*>(&cf[r][0]);
      const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
      const float2 v01 = make_float2(v4.x, v4.y), v23 = make_float2(v4.z, v4.w);
      const float2 w0 = make_float2(w.x, w.x), w1 = make_float2(w.y, w.y), w2 = make_float2(w.z, w.z);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 ki = make_float2(kk[i], kk[i]);
        const float2 kv[2] = {__fmul2_rn(ki, v01), __fmul2_rn(ki, v23)};
#pragma unroll
        for (int jp = 0; jp < 2; ++jp) {
          float2 a0 = make_float2(st[0][i][2 * jp], st[0][i][2 * jp + 1]);
          float2 a1 = make_float2(st[1][i][2 * jp], st[1][i][2 * jp + 1]);
          float2 a2 = make_float2(st[2][i][2 * jp], st[2][i][2 * jp + 1]);
          a0 = __ffma2_rn(w0, kv[jp], a0);
          a1 = __ffma2_rn(w1, kv[jp], a1);
          a2 = __ffma2_rn(w2, kv[jp], a2);
          st[0][i][2 * jp] = a0.x; st[0][i][2 * jp + 1] = a0.y;
          st[1][i][2 * jp] = a1.x; st[1][i][2 * jp + 1] = a1.y;
          st[2][i][2 * jp] = a2.x; st[2][i][2 * jp + 1] = a2.y;
        }
      }
    }
    __syncthreads();
  }
}

// ================================================================== chunk gradients
struct ChunkSmem {
  static constexpr uint32_t TILE = kCk * kLD;  // floats
  static constexpr int NTILE = 6;              // Q, K, V, dO, two product / state tiles
  static constexpr int NSC = 15;               // per-token scalar arrays
  // tiles, scalars, column partial sums [2][8 warps][kCk]; two CTAs fit on one SM
  static constexpr uint32_t BYTES = (NTILE * TILE + NSC * kCk + 8 * kCk * 2) * 4;
  static_assert(2 * (BYTES + 1024) <= 233472, "two CTAs per SM");
};

template <typename T>
__global__ void __launch_bounds__(kNT, 2) bwd_chunk_kernel(BwdArgs a, BwdChunkScratch scr) {
  extern __shared__ __align__(16) float sm[];
  float* Qs = sm;                       // q_hat rows (rotated unit vectors)
  float* Ks = Qs + ChunkSmem::TILE;     // k_hat rows
  float* Vs = Ks + ChunkSmem::TILE;     // v rows
  float* Ds = Vs + ChunkSmem::TILE;     // do rows
  float* P1 = Ds + ChunkSmem::TILE;     // A, then a state matrix, then dq_hat
  float* P2 = P1 + ChunkSmem::TILE;     // dC, then a state matrix, then dk_hat
  float* scal = P2 + ChunkSmem::TILE;   // [NSC][kCk]
  float* colp = scal + ChunkSmem::NSC * kCk;  // [2][8][kCk] column partials (one per warp)
  float* s_s = scal + 0 * kCk;    // s
  float* s_e = scal + 1 * kCk;    // e^{s - M_c}
  float* s_ah = scal + 2 * kCk;   // alpha~ e^{M_c - m}
  float* s_be = scal + 3 * kCk;   // beta
  float* s_ga = scal + 4 * kCk;   // gamma
  float* s_rho = scal + 5 * kCk;  // alpha~ e^{M_{c-1} - m}
  float* s_nq = scal + 6 * kCk;   // |q|
  float* s_nk = scal + 7 * kCk;   // |k|
  float* r_dah = scal + 8 * kCk;  // row sums: d ah (intra), d beta, d gamma
  float* r_dbe = scal + 9 * kCk;
  float* r_dga = scal + 10 * kCk;
  float* r_drho = scal + 11 * kCk;  // inter: d rho, d beta, d gamma
  float* r_dbe2 = scal + 12 * kCk;
  float* r_dga2 = scal + 13 * kCk;
  float* c_ds = scal + 14 * kCk;    // inter ds (e v.Z_F + v.Z_G)

  const int N = a.N, NC = (N + kCk - 1) / kCk;
  const int c = (int)(blockIdx.x % (unsigned)NC), bh = (int)(blockIdx.x / (unsigned)NC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tr = tid >> 4, tc = tid & 15;
  const size_t row0 = (size_t)bh * N;
  const int t0 = c * kCk, tn = min(N, t0 + kCk) - t0;
  const T* __restrict__ v = static_cast<const T*>(a.v) + row0 * kD;
  const T* __restrict__ dout = static_cast<const T*>(a.dout) + row0 * kD;
  const float Mc = scr.m[row0 + t0 + tn - 1];
  const float Mp = c > 0 ? scr.m[row0 + t0 - 1] : 0.0f;

  // ---- rows of the chunk (zero past N) and per-token scalars ----
  for (int r = warp; r < kCk; r += kNT / 32) {
    if (r < tn) {
      const size_t rw = row0 + t0 + r;
      Qs[r * kLD + lane] = scr.qhat[rw * kD + lane];
      Qs[r * kLD + lane + 32] = scr.qhat[rw * kD + lane + 32];
      Ks[r * kLD + lane] = scr.khat[rw * kD + lane];
      Ks[r * kLD + lane + 32] = scr.khat[rw * kD + lane + 32];
      const float nq = scr.nq[rw], nk = scr.nk[rw];
      Vs[r * kLD + lane] = ld(v, (size_t)(t0 + r) * kD + lane);
      Vs[r * kLD + lane + 32] = ld(v, (size_t)(t0 + r) * kD + lane + 32);
      Ds[r * kLD + lane] = ld(dout, (size_t)(t0 + r) * kD + lane);
      Ds[r * kLD + lane + 32] = ld(dout, (size_t)(t0 + r) * kD + lane + 32);
      if (lane == 0) {
        s_nq[r] = nq;
        s_nk[r] = nk;
      }
    } else {
      Qs[r * kLD + lane] = Qs[r * kLD + lane + 32] = 0.0f;
      Ks[r * kLD + lane] = Ks[r * kLD + lane + 32] = 0.0f;
      Vs[r * kLD + lane] = Vs[r * kLD + lane + 32] = 0.0f;
      Ds[r * kLD + lane] = Ds[r * kLD + lane + 32] = 0.0f;
      if (lane == 0) s_nq[r] = s_nk[r] = 1.0f;
    }
  }
  if (tid < kCk) {
    float sv = 0.0f, ev = 0.0f, ah = 0.0f, be = 0.0f, ga = 0.0f, rho = 0.0f;
    if (tid < tn) {
      const size_t row = row0 + t0 + tid;
      sv = scr.s[row];
      const float mt = scr.m[row];
      const TokCoef kc = tok_coef(a, row, t0 + tid, scr.E[row], scr.P[row]);
      ev = expf(__fsub_rn(sv, Mc));
      ah = __fmul_rn(kc.alt, expf(__fsub_rn(Mc, mt)));
      be = kc.beta;
      ga = kc.gamma;
      rho = c > 0 ? __fmul_rn(kc.alt, expf(__fsub_rn(Mp, mt))) : 0.0f;
    }
    s_s[tid] = sv;
    s_e[tid] = ev;
    s_ah[tid] = ah;
    s_be[tid] = be;
    s_ga[tid] = ga;
    s_rho[tid] = rho;
  }
  __syncthreads();

  // ---- intra-chunk products ----
  float dq[4][4], dk[4][4], dv[4][4];
  {
    float sa[4][4], da[4][4];
    zero44(sa);
    zero44(da);
    gemm64<false, true>(Qs, Ks, sa);  // S = Q K^T
    gemm64<false, true>(Ds, Vs, da);  // dA = dO V^T
    float rs_e[4], rs_s[4], rs_1[4], cp_a[4], cp_b[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) rs_e[x] = rs_s[x] = rs_1[x] = cp_a[x] = cp_b[x] = 0.0f;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int t = tr + 16 * x;
      const float ah = s_ah[t], be = s_be[t], ga = s_ga[t];
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const int i = tc + 16 * y;
        float av = 0.0f, dc = 0.0f;
        if (i <= t) {
          const float w = __fmaf_rn(ah, s_e[i], __fmaf_rn(be, s_s[i], ga));
          av = __fmul_rn(sa[x][y], w);
          dc = __fmul_rn(da[x][y], w);
          const float dw = __fmul_rn(da[x][y], sa[x][y]);
          rs_e[x] = __fmaf_rn(dw, s_e[i], rs_e[x]);
          rs_s[x] = __fmaf_rn(dw, s_s[i], rs_s[x]);
          rs_1[x] = __fadd_rn(rs_1[x], dw);
          cp_a[y] = __fmaf_rn(dw, ah, cp_a[y]);
          cp_b[y] = __fmaf_rn(dw, be, cp_b[y]);
        }
        P1[t * kLD + i] = av;
        P2[t * kLD + i] = dc;
      }
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const float e = sum16(rs_e[x]), s = sum16(rs_s[x]), o = sum16(rs_1[x]);
      if (tc == 0) {
        r_dah[tr + 16 * x] = e;
        r_dbe[tr + 16 * x] = s;
        r_dga[tr + 16 * x] = o;
      }
    }
#pragma unroll
    for (int y = 0; y < 4; ++y) {  // the warp's two row groups, then one partial per warp
      const float pa = cp_a[y] + __shfl_xor_sync(0xffffffffu, cp_a[y], 16);
      const float pb = cp_b[y] + __shfl_xor_sync(0xffffffffu, cp_b[y], 16);
      if (lane < 16) {
        colp[warp * kCk + tc + 16 * y] = pa;
        colp[8 * kCk + warp * kCk + tc + 16 * y] = pb;
      }
    }
  }
  __syncthreads();
  zero44(dq);
  zero44(dk);
  zero44(dv);
  gemm64<false, false>(P2, Ks, dq);  // dQ = dC K
  gemm64<true, false>(P2, Qs, dk);   // dK = dC^T Q
  gemm64<true, false>(P1, Ds, dv);   // dV = A^T dO
  float cA = 0.0f, cB = 0.0f;        // column sums of dW ah and dW beta (thread tid < 64)
  if (tid < kCk) {
    for (int g = 0; g < 8; ++g) {
      cA = __fadd_rn(cA, colp[g * kCk + tid]);
      cB = __fadd_rn(cB, colp[8 * kCk + g * kCk + tid]);
    }
  }
  __syncthreads();

  // ---- inter-chunk: the chunk-start states, X = dO M^T ----
  const float* fs = scr.fs + (((size_t)bh * NC + c) * 3) * kD * kD;
  const float* dsu = scr.ds + (((size_t)bh * NC + c) * 3) * kD * kD;
  for (int mtx = 0; mtx < 3; ++mtx) {
    float* Ms = (mtx & 1) ? P2 : P1;
    for (int e = tid; e < kD * kD / 4; e += kNT) {
      const float4 x4 = reinterpret_cast<const float4*>(fs + (size_t)mtx * kD * kD)[e];
      const int r = (4 * e) / kD, cc = (4 * e) % kD;
      *reinterpret_cast<float4*>(Ms + r * kLD + cc) = x4;
    }
    __syncthreads();
    float xa[4][4];
    zero44(xa);
    gemm64<false, true>(Ds, Ms, xa);  // X[t][a] = sum_j do_t[j] M[a][j]
    const float* coef = mtx == 0 ? s_rho : mtx == 1 ? s_be : s_ga;
    float* rdst = mtx == 0 ? r_drho : mtx == 1 ? r_dbe2 : r_dga2;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int t = tr + 16 * x;
      const float cf = coef[t];
      float rd = 0.0f;
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        dq[x][y] = __fmaf_rn(cf, xa[x][y], dq[x][y]);
        rd = __fmaf_rn(xa[x][y], Qs[t * kLD + tc + 16 * y], rd);
      }
      rd = sum16(rd);
      if (tc == 0) rdst[t] = rd;
    }
    __syncthreads();
  }

  // ---- suffix states: Y = V D^T (dk), Z = K D (dv, ds) ----
  float dsp[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // this thread's partial of e v.Z_F + v.Z_G per row
  for (int mtx = 0; mtx < 3; ++mtx) {
    float* Ms = (mtx & 1) ? P2 : P1;
    for (int e = tid; e < kD * kD / 4; e += kNT) {
      const float4 x4 = reinterpret_cast<const float4*>(dsu + (size_t)mtx * kD * kD)[e];
      const int r = (4 * e) / kD, cc = (4 * e) % kD;
      *reinterpret_cast<float4*>(Ms + r * kLD + cc) = x4;
    }
    __syncthreads();
    float ya[4][4], za[4][4];
    zero44(ya);
    zero44(za);
    gemm64<false, true>(Vs, Ms, ya);   // Y[i][a] = sum_j v_i[j] D[a][j]
    gemm64<false, false>(Ks, Ms, za);  // Z[i][j] = sum_a k_i[a] D[a][j]
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int i = tr + 16 * x;
      const float w = mtx == 0 ? s_e[i] : mtx == 1 ? s_s[i] : 1.0f;
      float rd = 0.0f;
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        dk[x][y] = __fmaf_rn(w, ya[x][y], dk[x][y]);
        dv[x][y] = __fmaf_rn(w, za[x][y], dv[x][y]);
        rd = __fmaf_rn(za[x][y], Vs[i * kLD + tc + 16 * y], rd);
      }
      if (mtx == 0) dsp[x] = __fmul_rn(s_e[i], rd);
      if (mtx == 1) dsp[x] = __fadd_rn(dsp[x], rd);
    }
    __syncthreads();
  }
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const float r = sum16(dsp[x]);
    if (tc == 0) c_ds[tr + 16 * x] = r;
  }

  // ---- outputs: dv directly; dq_hat, dk_hat staged for the unit-vector backward ----
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int t = tr + 16 * x;
    if (t < tn) {
#pragma unroll
      for (int y = 0; y < 4; ++y) a.dv[(row0 + t0 + t) * kD + tc + 16 * y] = dv[x][y];
    }
#pragma unroll
    for (int y = 0; y < 4; ++y) {
      P1[t * kLD + tc + 16 * y] = dq[x][y];
      P2[t * kLD + tc + 16 * y] = dk[x][y];
    }
  }
  __syncthreads();
  // dx = R^T (dy - y_hat (y_hat . dy)) / |x|, one warp per row (lane: the pair lane, lane + 32)
  for (int r = warp; r < tn; r += kNT / 32) {
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const float* dy = (which ? P2 : P1) + r * kLD;
      const float* yh = (which ? Ks : Qs) + r * kLD;
      float g0 = dy[lane], g1 = dy[lane + 32];
      float dot = __fmaf_rn(yh[lane], g0, __fmul_rn(yh[lane + 32], g1));
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) dot = __fadd_rn(dot, __shfl_xor_sync(0xffffffffu, dot, o));
      g0 = __fsub_rn(g0, __fmul_rn(yh[lane], dot));
      g1 = __fsub_rn(g1, __fmul_rn(yh[lane + 32], dot));
      if (a.rope) {  // inverse rotation of the pair
        const float2 cs = a.rope_table[(size_t)(t0 + r) * (kD / 2) + lane];
        const float x0 = __fmaf_rn(g0, cs.x, __fmul_rn(g1, cs.y));
        const float x1 = __fmaf_rn(-g0, cs.y, __fmul_rn(g1, cs.x));
        g0 = x0;
        g1 = x1;
      }
      const float inv = __fdiv_rn(1.0f, which ? s_nk[r] : s_nq[r]);
      float* dst = (which ? a.dk : a.dq) + (row0 + t0 + r) * kD;
      dst[lane] = __fmul_rn(g0, inv);
      dst[lane + 32] = __fmul_rn(g1, inv);
    }
  }
  // ---- per-token scalars: d alpha~, d gamma, direct ds; gate gradients ----
  if (tid < tn) {
    const int t = tid;
    const size_t row = row0 + t0 + t;
    const float mt = scr.m[row];
    const float dal = __fadd_rn(__fmul_rn(r_dah[t], expf(__fsub_rn(Mc, mt))),
                                c > 0 ? __fmul_rn(r_drho[t], expf(__fsub_rn(Mp, mt))) : 0.0f);
    const float dbe = __fadd_rn(r_dbe[t], r_dbe2[t]);
    const float dga = __fadd_rn(r_dga[t], r_dga2[t]);
    const float dsd = __fadd_rn(__fmaf_rn(s_e[t], cA, cB), c_ds[t]);
    float* tk = scr.tok + row * 4;
    tk[0] = dal;
    tk[1] = dga;
    tk[2] = dsd;
    const float Et = scr.E[row], P = scr.P[row];
    const float sig1 = sigmoid(a.g1[row]), sigh = sigmoid(a.gh[row]);
    const float rt = __fdiv_rn(1.0f, (float)(t0 + t + 1));
    const float Pt2 = __fmul_rn(__fmul_rn(P, rt), rt);
    const float dsig1 = __fsub_rn(__fmul_rn(dbe, rt), __fmul_rn(dga, Pt2));
    const float dsigh = __fadd_rn(__fsub_rn(__fdiv_rn(dal, Et), __fmul_rn(dbe, rt)),
                                  __fmul_rn(dga, __fsub_rn(Pt2, rt)));
    a.dg1[row] = __fmul_rn(dsig1, __fmul_rn(sig1, __fsub_rn(1.0f, sig1)));
    a.dgh[row] = __fmul_rn(dsigh, __fmul_rn(sigh, __fsub_rn(1.0f, sigh)));
    if (a.g0 && a.dg0) {
      const float s0 = sigmoid(a.g0[row]);
      a.dg0[row] = __fmul_rn(__fmul_rn(dga, rt), __fmul_rn(s0, __fsub_rn(1.0f, s0)));
    }
  }
}

// ================================================================== token scans
// ds_t = direct_t + e^{s_t - m_t} EA_t + PA_t with the suffix recurrences
// EA_t = e^{m_t - m_{t+1}} EA_{t+1} - alpha~_t d alpha~_t / E~_t and PA_t = PA_{t+1} -
// (beta_t / t) d gamma_t (the E and P terms of ds, as in the token-sequential kernel).  One CTA
// per (b, h); thread i takes a segment of consecutive tokens: it composes its segment's affine
// map EA_in -> EA_out, a single thread chains the segments from the end, then every thread
// replays its segment from its carry.
__global__ void __launch_bounds__(kNT) bwd_ds_kernel(BwdArgs a, BwdChunkScratch scr) {
  __shared__ float segR[kNT], segB[kNT], segP[kNT];  // segment maps, then carries
  const int bh = blockIdx.x, N = a.N, tid = threadIdx.x;
  const size_t row0 = (size_t)bh * N;
  const int L = (N + kNT - 1) / kNT, ta = min(N, tid * L), tb = min(N, ta + L);
  auto coef = [&](int t, float& r, float& b, float& p, float& ex) {
    const size_t row = row0 + t;
    const float* tk = scr.tok + row * 4;
    const float Et = scr.E[row], m = scr.m[row];
    const float sig1 = sigmoid(a.g1[row]), sigh = sigmoid(a.gh[row]);
    const float tf = (float)(t + 1);
    const float alt = __fdiv_rn(sigh, Et);
    const float beta = __fmul_rn(__fsub_rn(sig1, sigh), __fdiv_rn(1.0f, tf));
    b = -__fdiv_rn(__fmul_rn(alt, tk[0]), Et);
    p = -__fmul_rn(__fdiv_rn(beta, tf), tk[1]);
    r = t + 1 < N ? expf(__fsub_rn(m, scr.m[row + 1])) : 0.0f;
    ex = expf(__fsub_rn(scr.s[row], m));
  };
  // EA_ta = R EA_tb + B over the segment (tokens tb-1 down to ta)
  float R = 1.0f, B = 0.0f, PS = 0.0f;
  for (int t = tb - 1; t >= ta; --t) {
    float r, b, p, ex;
    coef(t, r, b, p, ex);
    B = __fmaf_rn(B, r, b);
    R = __fmul_rn(R, r);
    PS = __fadd_rn(PS, p);
  }
  segR[tid] = R;
  segB[tid] = B;
  segP[tid] = PS;
  __syncthreads();
  if (tid == 0) {  // carries: EA and PA entering each segment from the tokens after it
    float ea = 0.0f, pa = 0.0f;
    for (int g = kNT - 1; g >= 0; --g) {
      const float r = segR[g], b = segB[g], p = segP[g];
      segR[g] = ea;
      segB[g] = pa;
      ea = __fmaf_rn(ea, r, b);
      pa = __fadd_rn(pa, p);
    }
  }
  __syncthreads();
  float EA = segR[tid], PA = segB[tid];
  for (int t = tb - 1; t >= ta; --t) {
    float r, b, p, ex;
    coef(t, r, b, p, ex);
    EA = __fmaf_rn(EA, r, b);
    PA = __fadd_rn(PA, p);
    float* tk = scr.tok + (row0 + t) * 4;
    tk[3] = __fadd_rn(tk[2], __fmaf_rn(ex, EA, PA));
  }
}

// ubar (prefix of u), Z (suffix of ds u / (e^tau + t)), du = -(ds ubar + Z)/sqrt d and the d tau
// partial sums.  Grid (b h, column groups of 16): 64 token segments x 16 columns per CTA, the
// segments' totals combined through shared memory.
constexpr int kSeg = 64, kCols = 16;
template <typename T>
__global__ void __launch_bounds__(kSeg * kCols) bwd_du_kernel(BwdArgs a, BwdChunkScratch scr) {
  __shared__ float segu[kSeg][kCols], segz[kSeg][kCols];
  __shared__ float red[kSeg * kCols / 32];
  const int bh = blockIdx.x, h = bh % a.H;
  const int N = a.N, tid = threadIdx.x;
  const size_t row0 = (size_t)bh * N;
  const float etau = expf(a.tau[h]);
  const float rsd = __fdiv_rn(1.0f, __fsqrt_rn((float)kD));
  const T* __restrict__ u = static_cast<const T*>(a.u) + row0 * kD;
  const int g = tid / kCols, jj = tid % kCols, j = blockIdx.y * kCols + jj;
  const int L = (N + kSeg - 1) / kSeg, ta = min(N, g * L), tb = min(N, ta + L);
  const float mu = a.mu[(size_t)h * kD + j];
  float su = 0.0f;
#pragma unroll 4
  for (int t = ta; t < tb; ++t) su = __fadd_rn(su, ld(u, (size_t)t * kD + j));
  segu[g][jj] = su;
  __syncthreads();
  float S = 0.0f;
  for (int x = 0; x < g; ++x) S = __fadd_rn(S, segu[x][jj]);
  const float emu = __fmul_rn(etau, mu);
  float zl = 0.0f;
#pragma unroll 4
  for (int t = ta; t < tb; ++t) {
    const float ut = ld(u, (size_t)t * kD + j);
    S = __fadd_rn(S, ut);
    const float wt = __fdiv_rn(1.0f, __fadd_rn(etau, (float)(t + 1)));
    scr.ubar[(row0 + t) * kD + j] = __fmul_rn(__fadd_rn(emu, S), wt);
    zl = __fmaf_rn(__fmul_rn(scr.tok[(row0 + t) * 4 + 3], ut), wt, zl);
  }
  segz[g][jj] = zl;
  __syncthreads();
  float z = 0.0f;
  for (int x = g + 1; x < kSeg; ++x) z = __fadd_rn(z, segz[x][jj]);
  float tacc = 0.0f;
#pragma unroll 4
  for (int t = tb - 1; t >= ta; --t) {
    const float ut = ld(u, (size_t)t * kD + j);
    const float ds = scr.tok[(row0 + t) * 4 + 3];
    const float ub = scr.ubar[(row0 + t) * kD + j];
    const float wt = __fdiv_rn(1.0f, __fadd_rn(etau, (float)(t + 1)));
    const float dsu = __fmul_rn(ds, ut);
    z = __fmaf_rn(dsu, wt, z);
    tacc = __fmaf_rn(__fmul_rn(dsu, __fsub_rn(mu, ub)), wt, tacc);
    a.du[(row0 + t) * kD + j] = -__fmul_rn(__fmaf_rn(ds, ub, z), rsd);
  }
  // d mu: Z at the first token (segment 0 ends with the total); d tau: every partial
  if (g == 0) atomicAdd(a.dmu + (size_t)h * kD + j, -__fmul_rn(__fmul_rn(etau, z), rsd));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) tacc = __fadd_rn(tacc, __shfl_xor_sync(0xffffffffu, tacc, o));
  if ((tid & 31) == 0) red[tid >> 5] = tacc;
  __syncthreads();
  if (tid == 0) {
    float ts = 0.0f;
    for (int w = 0; w < kSeg * kCols / 32; ++w) ts = __fadd_rn(ts, red[w]);
    atomicAdd(a.dtau + h, -__fmul_rn(__fmul_rn(etau, ts), rsd));
  }
}

template <typename T>
cudaError_t launch_chunk_t(const BwdArgs& a, const BwdChunkScratch& sc, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(bwd_chunk_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)ChunkSmem::BYTES);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  const int BH = a.B * a.H, NC = (a.N + kCk - 1) / kCk;
  const size_t warps = 2 * (size_t)BH * a.N;
  const size_t rb = (warps * 32 + kNT - 1) / kNT;
  bwd_rows_kernel<T><<<(unsigned)(rb < 152 * 32 ? rb : 152 * 32), kNT, 0, stream>>>(a, sc);
  bwd_states_kernel<T><<<dim3(BH, 1, 2), kNT, 0, stream>>>(a, sc);
  bwd_chunk_kernel<T><<<(unsigned)(BH * NC), kNT, ChunkSmem::BYTES, stream>>>(a, sc);
  bwd_ds_kernel<<<BH, kNT, 0, stream>>>(a, sc);
  bwd_du_kernel<T><<<dim3(BH, kD / kCols), kSeg * kCols, 0, stream>>>(a, sc);
  count_launches(5);
  return cudaGetLastError();
}

}  // namespace

bool bwd_chunk_supported(int d) { return d == kD; }

// Scratch (bytes) of the chunked backward: forward scalars s, E e^{-m}, P, m [BH][N] each (the
// forward kernels write them first), chunk-start and suffix states, token scalars, prior means.
size_t bwd_chunk_scratch_bytes(int B, int H, int N, int d) {
  const size_t BH = (size_t)B * H, NC = (size_t)(N + kCk - 1) / kCk;
  return (BH * N * 4 + 2 * BH * NC * 3 * (size_t)d * d + BH * N * 4 + BH * N * (size_t)d +
          BH * N * (2 * (size_t)d + 2)) *
         sizeof(float);
}

cudaError_t launch_bwd_chunk(const BwdArgs& a, float* scratch, cudaStream_t stream) {
  const size_t BH = (size_t)a.B * a.H, N = (size_t)a.N, NC = (N + kCk - 1) / kCk;
  BwdChunkScratch sc;
  sc.s = scratch;
  sc.E = sc.s + BH * N;
  sc.P = sc.E + BH * N;
  sc.m = sc.P + BH * N;
  sc.fs = sc.m + BH * N;
  sc.ds = sc.fs + BH * NC * 3 * kD * kD;
  sc.tok = sc.ds + BH * NC * 3 * kD * kD;
  sc.ubar = sc.tok + BH * N * 4;
  sc.qhat = sc.ubar + BH * N * kD;
  sc.khat = sc.qhat + BH * N * kD;
  sc.nq = sc.khat + BH * N * kD;
  sc.nk = sc.nq + BH * N;
  return a.dtype == 1 ? launch_chunk_t<float>(a, sc, stream)
                      : launch_chunk_t<__nv_bfloat16>(a, sc, stream);
}

}  // namespace zs
