// Shared device code of the ZeroS GB300 library.
//
// The one numerics contract every kernel obeys (so that the logit s_t, the prefix sum P_t,
// the running maximum m_t and the scaled prefix sum Et_t = E_t e^{-m_t} come out bit-identical
// whether a sequence is processed by a forward kernel or token by token by the decode kernel):
//
//   for each new token t (1-based count), with d = 32 R and lane l of a warp owning the columns
//   a = l + 32 r (r = 0..R-1):
//     S[a]   <- S[a] + u_t[a]                          fp32, one add per column, token order
//     n[a]    = fma(e^tau, mu[a], S[a])                numerator of the prior mean times (e^tau+t)
//     p_l     = u[l]*n[l], then p_l = fma(u[l+32r], n[l+32r], p_l) for r = 1..R-1
//     dot     = butterfly sum of p_l over the lanes (xor offsets 16, 8, 4, 2, 1; own + partner)
//     s_t     = -dot / ((e^tau + t) * sqrt(d))
//     m_t     = max(m_{t-1}, s_t)                      (m_0 = -inf)
//     Et_t    = fma(Et_{t-1}, exp(m_{t-1} - m_t), exp(s_t - m_t))     (Et_0 = 0)
//     P_t     = P_{t-1} + s_t
//   every operation is an explicit round-to-nearest intrinsic (no contraction, no fast math),
//   and exp is CUDA's expf.  This is the deviation-logit definition of the Paper-Notes page
//   "ZeroS: Zero-Sum Linear Attention for Efficient Transformers" (method details, "deviation
//   logits": s_i = -(1/sqrt d) u_i ubar_i^T with ubar_i = (e^tau mu + sum_{j<=i} u_j)/(e^tau + i))
//   and its prefix sums E_t = sum e^{s_i}, P_t = sum s_i ("linear-time prefix scan"), evaluated
//   in one fixed fp32 order.  The running maximum keeps every exponential <= 1.
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
  float m;
  float Et;
  float P;
  float etau;
  float pad[3];
};
static_assert(sizeof(RecordHead) == 32, "record head is 32 bytes");

__host__ __device__ constexpr size_t record_bytes(int d) {
  return ((32 + 8 * (size_t)d + 12 * (size_t)d * d) + 255) / 256 * 256;
}
__host__ __device__ constexpr size_t state_bytes(int B, int H, int d) {
  return 256 + (size_t)B * H * record_bytes(d);
}
// Float offsets inside a record.
__host__ __device__ constexpr int rec_S(int) { return 8; }
__host__ __device__ constexpr int rec_mu(int d) { return 8 + d; }
__host__ __device__ constexpr int rec_F(int d) { return 8 + 2 * d; }
__host__ __device__ constexpr int rec_G(int d) { return 8 + 2 * d + d * d; }
__host__ __device__ constexpr int rec_H(int d) { return 8 + 2 * d + 2 * d * d; }

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

// Per-token scalar state carried by every path.
struct Scalars {
  float m;   // running maximum of s
  float Et;  // E_t * exp(-m_t)
  float P;   // sum of s
};

// The canonical token update above, executed by one full warp.  u, S, mu hold the lane's
// columns a = lane + 32 r.  Returns s_t (identical in every lane); updates S and sc in place
// (identical in every lane).  `t` is the 1-based token count including this token.
template <int R>
__device__ __forceinline__ float token_update(const float (&u)[R], float (&S)[R], const float (&mu)[R],
                                              float etau, int t, Scalars& sc, float* f_out,
                                              float* g_out) {
#pragma unroll
  for (int r = 0; r < R; ++r) S[r] = __fadd_rn(S[r], u[r]);
  float p = __fmul_rn(u[0], __fmaf_rn(etau, mu[0], S[0]));
#pragma unroll
  for (int r = 1; r < R; ++r) p = __fmaf_rn(u[r], __fmaf_rn(etau, mu[r], S[r]), p);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, o));
  const float den = __fmul_rn(__fadd_rn(etau, (float)t), __fsqrt_rn((float)(32 * R)));
  const float s = -__fdiv_rn(p, den);
  const float m_new = fmaxf(sc.m, s);
  const float f = expf(__fsub_rn(sc.m, m_new));
  const float g = expf(__fsub_rn(s, m_new));
  sc.Et = __fmaf_rn(sc.Et, f, g);
  sc.P = __fadd_rn(sc.P, s);
  sc.m = m_new;
  *f_out = f;
  *g_out = g;
  return s;
}

// Logit of one token against a fixed prior numerator n[a] (encoder mode: the full-sequence
// mean), same lane/tree order as token_update.
template <int R>
__device__ __forceinline__ float fixed_logit(const float (&u)[R], const float (&n)[R], float den) {
  float p = __fmul_rn(u[0], n[0]);
#pragma unroll
  for (int r = 1; r < R; ++r) p = __fmaf_rn(u[r], n[r], p);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, o));
  return -__fdiv_rn(p, den);
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

}  // namespace zs
