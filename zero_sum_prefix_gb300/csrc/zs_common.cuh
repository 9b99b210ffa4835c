// Shared device code of the ZeroS GB300 library.
//
// The one numerics contract every kernel obeys (so that the logit s_t, the prefix sum P_t,
// the running maximum m_t and the scaled prefix sum Et_t = E_t e^{-m_t} come out bit-identical
// whether a sequence is processed by a forward kernel or token by token by the decode step):
//
// Tokens are grouped in blocks of 32 (block b holds tokens 32b+1 .. 32b+32, t 1-based).  Every
// running quantity is a carry (its value at the end of the previous block) plus a local value
// accumulated inside the current block, so that the blocks of a chunk can be processed in
// parallel and then chained by one operation per block.  With d = 32 R and lane l of a warp
// owning the R contiguous columns a = R l + r:
//     L[a] <- L[a] + u_t[a]                 (local column sum, reset at each block start)
//     S[a]  = C[a] + L[a]                   (C = S at the end of the previous block)
//     n[a]  = fma(e^tau, mu[a], S[a])       (numerator of the prior mean times e^tau + t)
//     p_l   = u[Rl] n[Rl], then p_l = fma(u[Rl+r], n[Rl+r], p_l) for r = 1..R-1
//     dot   = butterfly sum of p_l over the lanes (xor offsets 16, 8, 4, 2, 1; own + partner)
//     s_t   = -dot / ((e^tau + t) sqrt(d))
//     LP   <- LP + s_t,        P_t = CP + LP
//     ml'   = max(ml, s_t),    El <- fma(El, exp(ml - ml'), exp(s_t - ml')),  ml <- ml'
//     m_t   = max(mC, ml),     Et_t = fma(EC, exp(mC - m_t), El exp(ml - m_t))
//     at a block's last token: C = S, CP = P_t, mC = m_t, EC = Et_t; L = 0, LP = 0,
//     ml = -inf, El = 0.
// Every operation is an explicit round-to-nearest intrinsic (no contraction, no fast math) and
// exp is CUDA's expf.  This evaluates the deviation logits of the Paper-Notes page "ZeroS:
// Zero-Sum Linear Attention for Efficient Transformers" (method details, "deviation logits":
// s_i = -(1/sqrt d) u_i ubar_i^T, ubar_i = (e^tau mu + sum_{j<=i} u_j)/(e^tau + i)) and the
// prefix sums E_t = sum e^{s_i}, P_t = sum s_i of its "linear-time prefix scan" in one fixed
// fp32 order; the running maximum keeps every exponential <= 1.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace zs {

enum : int {
  kOk = 0,
  kErrInvalid = 1,
  kErrUnsupported = 2,
  kErrRange = 3,
  kErrTimeout = 4,
  kErrCuda = 5
};

// Records the first device-side error of a launch sequence (later errors do not overwrite it).
__device__ __forceinline__ void report(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------------------------------------
// State blob layout (see include/zeros.h).
struct StateHeader {
  char magic[4];  // "ZSP1"
  int version;
  int B, H, d, dtype, rope;
  float rope_base;
  int pad[56];
};
static_assert(sizeof(StateHeader) == 256, "state header is 256 bytes");

struct RecordHead {  // first 32 bytes of every (b, h) record
  int t;
  float mC, EC, CP;  // carries at the end of the last completed block
  float etau;
  float ml, El, LP;  // local values of the current block
};
static_assert(sizeof(RecordHead) == 32, "record head is 32 bytes");

__host__ __device__ constexpr size_t record_bytes(int d) {
  return ((32 + 12 * (size_t)d + 12 * (size_t)d * d) + 255) / 256 * 256;
}
__host__ __device__ constexpr size_t state_bytes(int B, int H, int d) {
  return 256 + (size_t)B * H * record_bytes(d);
}
// Float offsets inside a record: C (column-sum carry), L (local column sums), mu, F~, G, H.
__host__ __device__ constexpr int rec_C(int) { return 8; }
__host__ __device__ constexpr int rec_L(int d) { return 8 + d; }
__host__ __device__ constexpr int rec_mu(int d) { return 8 + 2 * d; }
__host__ __device__ constexpr int rec_F(int d) { return 8 + 3 * d; }
__host__ __device__ constexpr int rec_G(int d) { return 8 + 3 * d + d * d; }
__host__ __device__ constexpr int rec_H(int d) { return 8 + 3 * d + 2 * d * d; }

__device__ __forceinline__ float* record_ptr(void* state, int bh, int d) {
  return reinterpret_cast<float*>(reinterpret_cast<char*>(state) + 256 + (size_t)bh * record_bytes(d));
}

// ------------------------------------------------------------------------------------------
// Element loads / stores for the two storage dtypes.
__device__ __forceinline__ float ld(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st(float* p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st(__nv_bfloat16* p, size_t i, float x) {
  p[i] = __float2bfloat16_rn(x);
}

// ------------------------------------------------------------------------------------------
// Gate: sigmoid of a gate logit (Paper-Notes, key design: "sigma_t^1, sigma_t^h are sigmoid
// gates that depend on the current step t").
__device__ __forceinline__ float sigmoid(float x) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-x)));
}

constexpr int kBlk = 32;  // block length of the numerics contract

// Running scalars of one sequence (identical in every lane of the owning warp).
struct Scalars {
  float mC, EC, CP;  // carries: m, Et and P at the end of the previous block
  float ml, El, LP;  // block-local running max, scaled exp-sum and logit sum
};

__device__ __forceinline__ Scalars scalars_init() {
  return Scalars{-INFINITY, 0.0f, 0.0f, -INFINITY, 0.0f, 0.0f};
}

// Logit dot product of one token, canonical lane/tree order (lane owns columns R l + r).
template <int R>
__device__ __forceinline__ float logit_dot(const float (&u)[R], const float (&n)[R]) {
  float p = __fmul_rn(u[0], n[0]);
#pragma unroll
  for (int r = 1; r < R; ++r) p = __fmaf_rn(u[r], n[r], p);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, o));
  return p;
}

// Per-token outputs of the contract.
struct TokenOut {
  float s, P, m, Et;
  float m_prev;  // m_{t-1} (running max before this token; -inf for the first token)
};

// The canonical token update, executed by one full warp.  u, C, L, mu hold the lane's columns
// R l + r.  `t` is the 1-based count including this token.  Updates C, L and sc in place.
template <int R>
__device__ __forceinline__ TokenOut token_update(const float (&u)[R], float (&C)[R], float (&L)[R],
                                                 const float (&mu)[R], float etau, int t,
                                                 Scalars& sc) {
  TokenOut o;
  o.m_prev = fmaxf(sc.mC, sc.ml);
  float S[R], n[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    L[r] = __fadd_rn(L[r], u[r]);
    S[r] = __fadd_rn(C[r], L[r]);
    n[r] = __fmaf_rn(etau, mu[r], S[r]);
  }
  const float dot = logit_dot<R>(u, n);
  const float den = __fmul_rn(__fadd_rn(etau, (float)t), __fsqrt_rn((float)(32 * R)));
  const float s = -__fdiv_rn(dot, den);
  sc.LP = __fadd_rn(sc.LP, s);
  const float P = __fadd_rn(sc.CP, sc.LP);
  const float ml = fmaxf(sc.ml, s);
  sc.El = __fmaf_rn(sc.El, expf(__fsub_rn(sc.ml, ml)), expf(__fsub_rn(s, ml)));
  sc.ml = ml;
  const float m = fmaxf(sc.mC, ml);
  const float Et = __fmaf_rn(sc.EC, expf(__fsub_rn(sc.mC, m)),
                             __fmul_rn(sc.El, expf(__fsub_rn(ml, m))));
  if ((t - 1) % kBlk == kBlk - 1) {  // block end: fold the local values into the carries
#pragma unroll
    for (int r = 0; r < R; ++r) {
      C[r] = S[r];
      L[r] = 0.0f;
    }
    sc.CP = P;
    sc.mC = m;
    sc.EC = Et;
    sc.LP = 0.0f;
    sc.ml = -INFINITY;
    sc.El = 0.0f;
  }
  o.s = s;
  o.P = P;
  o.m = m;
  o.Et = Et;
  return o;
}

// Logit of one token against a fixed prior numerator n[a] (encoder mode: the full-sequence
// mean), same lane/tree order as token_update.
template <int R>
__device__ __forceinline__ float fixed_logit(const float (&u)[R], const float (&n)[R], float den) {
  return -__fdiv_rn(logit_dot<R>(u, n), den);
}

// ------------------------------------------------------------------------------------------
// Rotary factors.  Angle = pos * base^(-2a/d) reduced modulo 2 pi in fp64, then sin/cos in
// fp32 of the reduced angle (error ~1e-7 at any position below 2^31).
__device__ __forceinline__ float2 rope_cs(double pos, int a, int d, double base) {
  const double theta = pow(base, -2.0 * (double)a / (double)d);
  const double ang = pos * theta;
  const double two_pi = 6.283185307179586476925286766559;
  const double r = ang - rint(ang / two_pi) * two_pi;
  float s, c;
  sincosf((float)r, &s, &c);
  return make_float2(c, s);
}

// Unit-normalise and (optionally) rotate one row held by a warp: lane l owns x[l + 32 r].
// Pairs are (a, a + d/2).  cs[r] = (cos, sin) for the pair index of column a = l + 32 r when
// that column is the first member of its pair (for d = 32 the partner lives in lane l ^ 16).
template <int R>
__device__ __forceinline__ void unit_rotate(float (&x)[R], bool rope, const float2 (&cs)[R]) {
  float ss = 0.0f;
#pragma unroll
  for (int r = 0; r < R; ++r) ss = __fmaf_rn(x[r], x[r], ss);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
  const float inv = __fdiv_rn(1.0f, fmaxf(__fsqrt_rn(ss), 1e-12f));
#pragma unroll
  for (int r = 0; r < R; ++r) x[r] = __fmul_rn(x[r], inv);
  if (!rope) return;
  const int lane = threadIdx.x & 31;
  if (R == 1) {
    // d = 32: pair (l, l + 16) lives in lanes l and l ^ 16.
    const float other = __shfl_xor_sync(0xffffffffu, x[0], 16);
    const float c = cs[0].x, s = cs[0].y;  // cs is the pair's factor in both lanes
    x[0] = (lane < 16) ? __fsub_rn(__fmul_rn(x[0], c), __fmul_rn(other, s))
                       : __fadd_rn(__fmul_rn(other, s), __fmul_rn(x[0], c));
  } else {
    constexpr int HALF = R / 2;  // column a = l + 32 r pairs with a + d/2 = l + 32 (r + HALF)
#pragma unroll
    for (int r = 0; r < HALF; ++r) {
      const float xa = x[r], xb = x[r + HALF];
      const float c = cs[r].x, s = cs[r].y;
      x[r] = __fsub_rn(__fmul_rn(xa, c), __fmul_rn(xb, s));
      x[r + HALF] = __fadd_rn(__fmul_rn(xa, s), __fmul_rn(xb, c));
    }
  }
}

// Pair index of lane's column r for head dimension d = 32 R.
template <int R>
__device__ __forceinline__ int pair_index(int lane, int r) {
  if (R == 1) return lane & 15;
  return lane + 32 * r;  // valid for r < R/2
}

// ------------------------------------------------------------------------ output LayerNorm
// Chan, Golub and LeVeque's pairwise update: merge the moments (count n, mean, M2 = sum of
// squared deviations) of one part of a row with those of another part (n2, mean2, m22).
__device__ __forceinline__ void moments_merge(float& n, float& mean, float& m2, float n2,
                                              float mean2, float m22) {
  const float nn = n + n2;
  const float delta = mean2 - mean;
  mean = __fmaf_rn(delta, n2 / nn, mean);
  m2 = m2 + m22 + delta * delta * (n * n2 / nn);
  n = nn;
}

// Sum over the 32 lanes of a warp (every lane receives it).
__device__ __forceinline__ float warp_sum32(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

}  // namespace zs
