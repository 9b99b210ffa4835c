// Encoder-mode (non-causal) ZeroS forward for d = 64, one CTA per (b, h) sequence.
//
// Method: Paper-Notes "ZeroS: Zero-Sum Linear Attention for Efficient Transformers", method
// details (deviation logits, zero-sum weights, radial-angular decoupling, linear-time prefix
// scan) and the training-strategy section (non-causal mode).  In encoder mode every sum runs
// over the whole sequence: the prior mean is the full-sequence mean, so every logit
// s_i = -(1/sqrt d) u_i ubar^T is independent of the others, and every output uses the same
// three states F = sum_i e^{s_i - m} k_hat_i^T v_i, G = sum_i s_i k_hat_i^T v_i,
// H = sum_i k_hat_i^T v_i (m the maximum logit):
//   o_t = q_hat_t (alpha~_t F + beta_t G + gamma_t H),  alpha~_t = sigh_t / E~,
//   beta_t = (sig1_t - sigh_t)/N,  gamma_t = -beta_t P/N - sigh_t/N (+ sig0_t/N),
// with E~ = sum_i e^{s_i - m} and P = sum_i s_i.  Nothing is sequential, so the kernel works in
// tiles of 64 tokens: a pass over the tokens for sum u, a pass accumulating the states in
// registers (each thread 3 x 16 state entries; the F state rescaled when the maximum grows), and
// a pass of 64 x 64 x 64 fp32 tile products Q [F|G|H] for the outputs, with the optional output
// LayerNorm fused.  Tiles are loaded with 16-byte vectors, four lanes per row.  All arithmetic fp32 (the token-sequential kernel remains the path that
// reports per-token debug scalars).
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

constexpr int kD = 64, kT = 64, kNT = 256, kLD = tiles::kLD;

struct EncSmem {
  static constexpr int TILE = kT * kLD;  // floats
  // rows (k_hat or q_hat), values, the three states, per-token arrays, reductions
  static constexpr int FLOATS = 2 * TILE + 3 * kD * kLD + 6 * kT + 4 * kD + 16;
  static constexpr unsigned BYTES = FLOATS * 4;
};

// Tile helpers: thread (r = tid / 4, quarter qq = tid % 4) owns columns 16 qq .. 16 qq + 15 of
// row r of a 64 x 64 tile (row stride kLD), so that every global load is a 16-byte vector and
// every row is handled by four neighbouring lanes.
template <typename T>
__device__ __forceinline__ void load16(const T* src, float (&x)[16]);
template <>
__device__ __forceinline__ void load16<float>(const float* src, float (&x)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 t = reinterpret_cast<const float4*>(src)[i];
    x[4 * i] = t.x; x[4 * i + 1] = t.y; x[4 * i + 2] = t.z; x[4 * i + 3] = t.w;
  }
}
template <>
__device__ __forceinline__ void load16<__nv_bfloat16>(const __nv_bfloat16* src, float (&x)[16]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 t = reinterpret_cast<const uint4*>(src)[i];
    const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[8 * i + 2 * e] = __uint_as_float(w[e] << 16);
      x[8 * i + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
  }
}

// Row r of the tile (zero past the sequence) into registers x; returns the row's squared norm
// (summed over the four lanes of the row).
template <typename T>
__device__ __forceinline__ float tile_row(const T* base, int t0, int tn, float (&x)[16]) {
  const int r = threadIdx.x >> 2, qq = threadIdx.x & 3;
  if (r < tn) {
    load16<T>(base + (size_t)(t0 + r) * kD + 16 * qq, x);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = 0.0f;
  }
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) ss = __fmaf_rn(x[i], x[i], ss);
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  ss += __shfl_xor_sync(0xffffffffu, ss, 2);
  return ss;
}

__device__ __forceinline__ void store_row(float* dst, const float (&x)[16]) {
  const int r = threadIdx.x >> 2, qq = threadIdx.x & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<float4*>(dst + r * kLD + 16 * qq + 4 * i) =
        make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
}

// Unit rows of a tile (rotated to their positions when rope): loads, normalises and stores; the
// rotation of the pairs (a, a + 32) runs after a barrier, thread (r, p) taking pairs 8p .. 8p + 7.
template <typename T>
__device__ __forceinline__ void unit_tile(const T* base, const FwdArgs& a, int t0, int tn,
                                          float* dst) {
  float x[16];
  const float ss = tile_row<T>(base, t0, tn, x);
  const float inv = __fdiv_rn(1.0f, fmaxf(__fsqrt_rn(ss), 1e-12f));
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] *= inv;
  store_row(dst, x);
  if (a.rope) {
    __syncthreads();
    const int r = threadIdx.x >> 2, p = threadIdx.x & 3;
    if (r < tn) {
      const float2* tab = a.rope_table + (size_t)(t0 + r) * (kD / 2) + 8 * p;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int c0 = 8 * p + e;
        const float2 cs = tab[e];
        const float x0 = dst[r * kLD + c0], x1 = dst[r * kLD + c0 + 32];
        dst[r * kLD + c0] = __fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, cs.y));
        dst[r * kLD + c0 + 32] = __fadd_rn(__fmul_rn(x0, cs.y), __fmul_rn(x1, cs.x));
      }
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kNT, 2) enc_kernel(FwdArgs a) {
  extern __shared__ __align__(16) float sm[];
  float* Rt = sm;                      // [kT][kLD] k_hat, then q_hat rows of a tile
  float* Vt = Rt + EncSmem::TILE;      // [kT][kLD] v rows of a tile
  float* Ms = Vt + EncSmem::TILE;      // [3][kD][kLD] F~, G, H
  float* ts = Ms + 3 * kD * kLD;       // [kT] s of the tile's tokens
  float* te = ts + kT;                 // [kT] e^{s - m}
  float* ca = te + kT;                 // [kT] alpha~, beta, gamma of the tile's rows
  float* cb = ca + kT;
  float* cg = cb + kT;
  float* red = cg + kT;                // [4][kD] column partial sums
  float* misc = red + 4 * kD;          // m, E~, P, rescale factor
  const int bh = blockIdx.x, h = bh % a.H;
  const int N = a.N, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t row0 = (size_t)bh * N;
  const T* __restrict__ q = static_cast<const T*>(a.q) + row0 * kD;
  const T* __restrict__ k = static_cast<const T*>(a.k) + row0 * kD;
  const T* __restrict__ v = static_cast<const T*>(a.v) + row0 * kD;
  const T* __restrict__ u = static_cast<const T*>(a.u) + row0 * kD;
  T* __restrict__ out = static_cast<T*>(a.out) + row0 * kD;
  const float etau = expf(a.tau[h]);

  // ---- full-sequence prior numerator n = e^tau mu + sum_j u_j ----
  {
    const int j = tid % kD, g = tid / kD;
    float su = 0.0f;
    for (int t = g; t < N; t += kNT / kD) su += ld(u, (size_t)t * kD + j);
    red[g * kD + j] = su;
  }
  if (tid == 0) {
    misc[0] = -INFINITY;  // running maximum m
    misc[1] = 0.0f;       // E~ = sum e^{s - m}
    misc[2] = 0.0f;       // P
  }
  __syncthreads();
  const float den = __fmul_rn(__fadd_rn(etau, (float)N), __fsqrt_rn((float)kD));
  __shared__ float nv[kD];  // numerator e^tau mu + sum_j u_j
  if (tid < kD) {
    float s0 = 0.0f;
    for (int g = 0; g < kNT / kD; ++g) s0 += red[g * kD + tid];
    nv[tid] = __fmaf_rn(etau, a.mu[(size_t)h * kD + tid], s0);
  }
  __syncthreads();

  // ---- states: thread owns row ar, columns cj .. cj + 15 of F~, G, H ----
  const int ar = tid >> 2, cj = (tid & 3) * 16;
  float sa[3][16];
#pragma unroll
  for (int m = 0; m < 3; ++m)
#pragma unroll
    for (int x = 0; x < 16; ++x) sa[m][x] = 0.0f;
  const int NT = (N + kT - 1) / kT;
  for (int c = 0; c < NT; ++c) {
    const int t0 = c * kT, tn = min(N, t0 + kT) - t0;
    unit_tile<T>(k, a, t0, tn, Rt);
    {
      float x[16];
      tile_row<T>(v, t0, tn, x);
      store_row(Vt, x);
      tile_row<T>(u, t0, tn, x);  // logits: s = -(u . n) / ((e^tau + N) sqrt d)
      const int r = tid >> 2, qq = tid & 3;
      float dot = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) dot = __fmaf_rn(x[i], nv[16 * qq + i], dot);
      dot += __shfl_xor_sync(0xffffffffu, dot, 1);
      dot += __shfl_xor_sync(0xffffffffu, dot, 2);
      if (qq == 0) ts[r] = r < tn ? -__fdiv_rn(dot, den) : -INFINITY;
    }
    __syncthreads();
    if (warp == 0) {  // tile maximum, new running maximum, E~ and P
      const float x0 = ts[lane], x1 = ts[lane + 32];
      float cm = fmaxf(x0, x1);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
      const float m_old = misc[0], m_new = fmaxf(m_old, cm);
      const float e0 = expf(__fsub_rn(x0, m_new)), e1 = expf(__fsub_rn(x1, m_new));
      te[lane] = e0;
      te[lane + 32] = e1;
      float es = e0 + e1;
      float ps = (lane < tn ? x0 : 0.0f) + (lane + 32 < tn ? x1 : 0.0f);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        es += __shfl_xor_sync(0xffffffffu, es, o);
        ps += __shfl_xor_sync(0xffffffffu, ps, o);
      }
      if (lane == 0) {
        const float f = m_old == -INFINITY ? 0.0f : expf(__fsub_rn(m_old, m_new));
        if (!isfinite(cm)) report(a.status, kErrRange);
        misc[0] = m_new;
        misc[1] = __fmaf_rn(misc[1], f, es);
        misc[2] += ps;
        misc[3] = f;
      }
    }
    __syncthreads();
    const float f = misc[3];
    if (f != 1.0f) {
#pragma unroll
      for (int x = 0; x < 16; ++x) sa[0][x] *= f;
    }
    for (int r = 0; r < tn; ++r) {
      const float kr = Rt[r * kLD + ar];
      const float we = te[r] * kr, wsv = ts[r] * kr;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const float4 vv = *reinterpret_cast<const float4*>(Vt + r * kLD + cj + 4 * q4);
        const float vx[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          sa[0][4 * q4 + e] = __fmaf_rn(we, vx[e], sa[0][4 * q4 + e]);
          sa[1][4 * q4 + e] = __fmaf_rn(wsv, vx[e], sa[1][4 * q4 + e]);
          sa[2][4 * q4 + e] = __fmaf_rn(kr, vx[e], sa[2][4 * q4 + e]);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int m = 0; m < 3; ++m)
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4)
      *reinterpret_cast<float4*>(Ms + m * kD * kLD + ar * kLD + cj + 4 * q4) =
          make_float4(sa[m][4 * q4], sa[m][4 * q4 + 1], sa[m][4 * q4 + 2], sa[m][4 * q4 + 3]);
  __syncthreads();
  const float Et = misc[1], P = misc[2];
  const float rN = __fdiv_rn(1.0f, (float)N);

  // ---- outputs: per tile of 64 queries, Q [F~|G|H] combined with the row coefficients ----
  const int tr = tid >> 4, tc = tid & 15;
  for (int c = 0; c < NT; ++c) {
    const int t0 = c * kT, tn = min(N, t0 + kT) - t0;
    unit_tile<T>(q, a, t0, tn, Rt);
    if (tid < kT) {
      float al = 0.0f, be = 0.0f, ga = 0.0f;
      if (tid < tn) {
        const size_t row = row0 + t0 + tid;
        const float sig1 = sigmoid(a.g1[row]), sigh = sigmoid(a.gh[row]);
        be = __fmul_rn(__fsub_rn(sig1, sigh), rN);
        ga = -__fadd_rn(__fmul_rn(__fmul_rn(be, P), rN), __fmul_rn(sigh, rN));
        if (a.g0) ga = __fadd_rn(ga, __fmul_rn(sigmoid(a.g0[row]), rN));
        al = __fdiv_rn(sigh, Et);
      }
      ca[tid] = al;
      cb[tid] = be;
      cg[tid] = ga;
    }
    __syncthreads();
    float o[4][4], x[4][4];
    zero44(o);
#pragma unroll 1
    for (int m = 0; m < 3; ++m) {
      zero44(x);
      gemm64<false, false>(Rt, Ms + m * kD * kLD, x);  // X[t][j] = sum_a q_hat_t[a] M[a][j]
      const float* cf = m == 0 ? ca : m == 1 ? cb : cg;
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int y = 0; y < 4; ++y) o[i][y] = __fmaf_rn(cf[tr + 16 * i], x[i][y], o[i][y]);
    }
    if (a.ln) {  // output LayerNorm over the row's 64 columns (16 threads x 4 columns)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float mean = sum16((o[i][0] + o[i][1]) + (o[i][2] + o[i][3])) * (1.0f / kD);
        float dv = 0.0f;
#pragma unroll
        for (int y = 0; y < 4; ++y) dv = __fmaf_rn(o[i][y] - mean, o[i][y] - mean, dv);
        const float rstd = rsqrtf(sum16(dv) * (1.0f / kD) + a.ln_eps);
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const int j = tc + 16 * y;
          const float w = a.ln_w ? a.ln_w[(size_t)h * kD + j] : 1.0f;
          const float b = a.ln_b ? a.ln_b[(size_t)h * kD + j] : 0.0f;
          o[i][y] = __fmaf_rn((o[i][y] - mean) * rstd, w, b);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = tr + 16 * i;
      if (t < tn) {
#pragma unroll
        for (int y = 0; y < 4; ++y) st(out, (size_t)(t0 + t) * kD + tc + 16 * y, o[i][y]);
      }
    }
    __syncthreads();
  }
}

}  // namespace

bool enc_supported(int d) { return d == kD; }

cudaError_t launch_fwd_encoder(const FwdArgs& a, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_set[2];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  const int f32 = a.dtype == 1;
  if (!(attr_set[f32].load() & bit)) {
    e = f32 ? cudaFuncSetAttribute(enc_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)EncSmem::BYTES)
            : cudaFuncSetAttribute(enc_kernel<__nv_bfloat16>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)EncSmem::BYTES);
    if (e != cudaSuccess) return e;
    attr_set[f32].fetch_or(bit);
  }
  if (f32)
    enc_kernel<float><<<a.B * a.H, kNT, EncSmem::BYTES, stream>>>(a);
  else
    enc_kernel<__nv_bfloat16><<<a.B * a.H, kNT, EncSmem::BYTES, stream>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace zs
