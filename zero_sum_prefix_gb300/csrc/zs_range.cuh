// Power-of-two range scales of the fp16 tensor-core operands of the chunked forward kernels.
//
// The operands (unit or unnormalised rotated q and k, S, the value-side tiles and the copy of
// the state) are fp16: eleven significant bits, against eight for bf16, with a range of
// about 6e-5 .. 65504 at full precision.  Each operand whose size grows with the data is
// multiplied by an exact power of two chosen from a bound of its entries, and the inverse
// power is folded into an fp32 coefficient of the product, so that no rounding is added:
//   * row t of S carries 2^kr_t with 2^kr_t |w_{t,i}| < 1 (the weights' bound);
//   * the state copy feeding chunk c carries 2^-kb_c with 2^kb_c > 128 c, the number of
//     tokens it sums (each entry is at most that many times max|v|: unit keys, e^{s - m} <= 1);
//   * G is accumulated with s 2^-ks, |s| 2^-ks < 1 over the sequence (the scalar pass writes the
//     largest |s| of each of its CTAs).
#pragma once

#include "zs_internal.h"

namespace zs {

// 2^k for |k| < 127 (exact).
__device__ __forceinline__ float pow2f(int k) { return __int_as_float((127 + k) << 23); }

// An exponent e with x < 2^e for x > 0 (the binary exponent of x plus one: 2^(e-1) <= x for
// normal x), 0 for x <= 0.
__device__ __forceinline__ int exp_above(float x) {
  return x > 0.0f ? (int)((__float_as_uint(x) >> 23) & 0xffu) - 126 : 0;
}

// kb of the state copy that feeds chunk c (chunks of `chunk` tokens).
__device__ __forceinline__ int state_exp(int c, int chunk) {
  return c > 0 ? exp_above((float)(c * chunk)) : 0;
}

// The sequence's largest |s| (from the scalar pass; 0 when not given).
__device__ __forceinline__ float seq_smax(const FwdArgs& a, int bh) {
  float m = 0.0f;
  if (a.smax) {
#pragma unroll
    for (int r = 0; r < kScalarCtas; ++r) m = fmaxf(m, __ldcg(a.smax + (size_t)bh * kScalarCtas + r));
  }
  return m;
}

// ks of the G products (at most 100).
__device__ __forceinline__ int s_exp(const FwdArgs& a, int bh) {
  return min(100, max(0, exp_above(seq_smax(a, bh))));
}

// kr of a row of S from the bound of its weights (clamped to |kr| <= 60).
__device__ __forceinline__ int row_exp(float wbound) {
  return min(60, max(-60, -exp_above(wbound)));
}

}  // namespace zs
