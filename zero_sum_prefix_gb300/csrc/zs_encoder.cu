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
#include "zs_sm100.cuh"
#include "zs_tiles.cuh"

namespace zs {
namespace {

using tiles::gemm64;
using tiles::sum16;
using tiles::zero44;
using namespace sm100;

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

// ============================================================== tensor-core encoder (bf16)
// The same computation with both contractions on tcgen05 (bf16 operands, fp32 accumulation in
// TMEM), one CTA of 256 threads per sequence.  Tiles of 128 tokens; token row r of a tile is
// TMEM lane r, handled by two threads (warps w and w + 4 share lane quadrant w & 3), each
// holding half of the row's columns:
//   states:  D1 = [e o v | s o v]^T K_hat  (M = 128: rows 0..63 = F~^T, 64..127 = G^T),
//            D2 = [v | e o v]^T K_hat       (rows 0..63 = H^T; the rest unused),
//            accumulated over the token tiles (A operands MN-major from the swizzled value
//            atoms, B = the k_hat atom, K = tokens);
//   outputs: D3 = Q_hat [F~ | G | H] (M = 128 tokens, N = 192, K = d), the states copied to a
//            K-major bf16 tile first, and o_t = alpha~_t D3_F + beta_t D3_G + gamma_t D3_H.
// The three terms nearly cancel (the weights sum to zero), so e o v, s o v and the states are
// each split into bf16 hi and lo parts (two products accumulated into one TMEM tile): only
// k_hat, q_hat and v, which the three terms share, are rounded to bf16 once.
// For q and k a thread takes the rotary pairs 16 hf .. 16 hf + 15 of its row (columns
// 16 hf + i and 32 + 16 hf + i), so that each rotation stays in one thread; the row's squared
// norm is the sum of the two halves (exchanged through shared memory).  For the states and the
// outputs it takes the contiguous columns 32 hf .. 32 hf + 31.
// Each token's logit is computed in one pass over u (the maximum, P and E~ together) and kept
// in shared memory for the state tiles when the sequence has at most 2048 tokens (recomputed
// otherwise).
constexpr int kTcThreads = 256, kTcT = 128, kTcNMax = 1 << 20;
constexpr uint32_t kAtom = 128 * 128;  // [128 rows x 64 bf16], 128-byte swizzle

struct EncTcSmem {
  // value atoms: v, then the hi and lo bf16 parts of e o v and s o v (the A operand pairs
  // [EVH | SVH] and [EVL | SVL] are contiguous), the k_hat / q_hat atom
  static constexpr uint32_t AV = 0, EVH = kAtom, SVH = 2 * kAtom, EVL = 3 * kAtom,
                            SVL = 4 * kAtom, KQ = 5 * kAtom;
  // [192 rows][64] K-major states, hi and lo bf16 parts: written after the last state product,
  // over the value atoms, which are dead by then (the q_hat atom KQ stays separate)
  static constexpr uint32_t BHI = 0;
  static constexpr uint32_t BLO = BHI + 192 * 128;
  static_assert(BLO + 192 * 128 <= KQ, "the state tiles overlay the value atoms only");
  // float [kD] prior numerator, then per warp: maximum, logit sum, exponential sum ([8] each)
  static constexpr uint32_t RED = 6 * kAtom;
  static constexpr uint32_t NRM = RED + (kD + 24) * 4;   // float [2][128]: half squared norms
  static constexpr uint32_t LNX = NRM + 2 * kTcT * 4;     // float2 [2][128]: half (mean, M2)
  static constexpr uint32_t BAR = LNX + 2 * kTcT * 8;     // mbarrier, TMEM address, abort flag
  // the logits of the first pass, kept for the state tiles when the sequence fits
  static constexpr int kSlogMax = 2048;
  static constexpr uint32_t SLOG = BAR + 64;
  static constexpr uint32_t BYTES = SLOG + kSlogMax * 4;
  static_assert(2 * (BYTES + 1024) <= 233472, "two CTAs per SM");
  static_assert(BAR % 8 == 0, "mbarrier alignment");
};

// The 16-byte chunk of the x-th eighth (0..3) of a thread's rotary-pair columns: chunks 2 hf,
// 2 hf + 1 (columns 16 hf ..) and 4 + 2 hf, 5 + 2 hf (their partners, + 32).
__device__ __forceinline__ int pair_chunk(int hf, int x) { return (x < 2 ? 2 * hf : 2 + 2 * hf) + x; }

// The raw bf16 words of this thread's rotary-pair columns of row t (loaded ahead of their use),
// and their values.
__device__ __forceinline__ void load_half_pairs(const __nv_bfloat16* row, bool valid, int hf,
                                                uint4 (&w)[4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    w[c] = valid ? reinterpret_cast<const uint4*>(row)[pair_chunk(hf, c)] : make_uint4(0u, 0u, 0u, 0u);
}
__device__ __forceinline__ void unpack_half(const uint4 (&w)[4], float (&x)[32]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    unpack_bf16x2(w[c].x, x[8 * c], x[8 * c + 1]);
    unpack_bf16x2(w[c].y, x[8 * c + 2], x[8 * c + 3]);
    unpack_bf16x2(w[c].z, x[8 * c + 4], x[8 * c + 5]);
    unpack_bf16x2(w[c].w, x[8 * c + 6], x[8 * c + 7]);
  }
}

__device__ __forceinline__ void put_half_pairs(uint8_t* atom, int r, int hf, const float (&x)[32]) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(atom + sw128_off(r, pair_chunk(hf, c))) =
        make_uint4(pack_bf16x2(x[8 * c], x[8 * c + 1]), pack_bf16x2(x[8 * c + 2], x[8 * c + 3]),
                   pack_bf16x2(x[8 * c + 4], x[8 * c + 5]), pack_bf16x2(x[8 * c + 6], x[8 * c + 7]));
}

// scale * x as the bf16 pair (hi, lo) with hi + lo = scale * x to about 2^-17 (the three state
// terms nearly cancel, so each is kept to fp32 accuracy), into the chunks chunk(c) of row r.
template <typename ChunkOf>
__device__ __forceinline__ void put_split(uint8_t* hi_atom, uint8_t* lo_atom, int r, float scale,
                                          const float (&x)[32], ChunkOf chunk) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t ph[4], pl[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float y0 = scale * x[8 * c + 2 * e], y1 = scale * x[8 * c + 2 * e + 1];
      const float h0 = __bfloat162float(__float2bfloat16_rn(y0));
      const float h1 = __bfloat162float(__float2bfloat16_rn(y1));
      ph[e] = pack_bf16x2(h0, h1);
      pl[e] = pack_bf16x2(y0 - h0, y1 - h1);
    }
    *reinterpret_cast<uint4*>(hi_atom + sw128_off(r, chunk(c))) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
    *reinterpret_cast<uint4*>(lo_atom + sw128_off(r, chunk(c))) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
  }
}

// Unit rotated half row: x scaled by 1 / max(|row|, 1e-12) (ss = the row's squared norm), then
// each of the thread's rotary pairs (x[i], x[16 + i]) = columns (16 hf + i, 32 + 16 hf + i)
// rotated to position t with rope.
__device__ __forceinline__ void unit_rot_half(const FwdArgs& a, int t, bool valid, int hf,
                                              float ss, float (&x)[32]) {
  const float inv = __fdiv_rn(1.0f, fmaxf(__fsqrt_rn(ss), 1e-12f));
#pragma unroll
  for (int i = 0; i < 32; ++i) x[i] *= inv;
  if (a.rope && valid) {
    const float2* tab = a.rope_table + (size_t)t * (kD / 2) + 16 * hf;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 cs = tab[i];
      const float x0 = x[i], x1 = x[16 + i];
      x[i] = __fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, cs.y));
      x[16 + i] = __fadd_rn(__fmul_rn(x0, cs.y), __fmul_rn(x1, cs.x));
    }
  }
}

__global__ void __launch_bounds__(kTcThreads, 2) enc_tc_kernel(FwdArgs a) {
  using SM = EncTcSmem;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) report(a.status, kErrUnsupported);
    return;
  }
  float* red = reinterpret_cast<float*>(smem + SM::RED);
  float* nrm = reinterpret_cast<float*>(smem + SM::NRM);
  float2* lnx = reinterpret_cast<float2*>(smem + SM::LNX);
  float* slog = reinterpret_cast<float*>(smem + SM::SLOG);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + SM::BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + SM::BAR + 8);
  int* abort_flag = reinterpret_cast<int*>(smem + SM::BAR + 12);
  const int bh = blockIdx.x, h = bh % a.H;
  const int N = a.N, tid = threadIdx.x, warp = tid >> 5;
  const int r = 32 * (warp & 3) + (tid & 31);  // token row of a tile = TMEM lane
  const int hf = warp >> 2;                    // which half of the row this thread holds
  const size_t row0 = (size_t)bh * N;
  const __nv_bfloat16* __restrict__ q = static_cast<const __nv_bfloat16*>(a.q) + row0 * kD;
  const __nv_bfloat16* __restrict__ k = static_cast<const __nv_bfloat16*>(a.k) + row0 * kD;
  const __nv_bfloat16* __restrict__ v = static_cast<const __nv_bfloat16*>(a.v) + row0 * kD;
  const __nv_bfloat16* __restrict__ u = static_cast<const __nv_bfloat16*>(a.u) + row0 * kD;
  __nv_bfloat16* __restrict__ out = static_cast<__nv_bfloat16*>(a.out) + row0 * kD;
  const float etau = expf(a.tau[h]);
  if (tid == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
  }
  if (warp == 0) {
    tmem_alloc(tslot, 256);
    tmem_relinquish();
  }
  // the first state tile's k and v words, loaded now: their latency passes under the two
  // passes over u; every later tile's are loaded while the previous tile's products run
  uint4 kw[4], vw[4];
  load_half_pairs(k + (size_t)r * kD, r < N, hf, kw);
  load_half_pairs(v + (size_t)r * kD, r < N, hf, vw);
  // ---- prior numerator: thread (p, g) sums columns 8 g .. 8 g + 7 over the tokens p, p + 32,
  //      ... with 16-byte loads (four rows in flight); the 32 partial sums of a column are then
  //      added by one thread (the q_hat atom, not used yet, holds them) ----
  {
    const int g = tid & 7, p = tid >> 3;
    float su[8];
#pragma unroll
    for (int y = 0; y < 8; ++y) su[y] = 0.0f;
    const uint4* ur = reinterpret_cast<const uint4*>(u) + g;
    auto add_row = [&](const uint4& w) {
      const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        float lo, hi;
        unpack_bf16x2(wv[y], lo, hi);
        su[2 * y] += lo;
        su[2 * y + 1] += hi;
      }
    };
    int t = p;
    for (; t + 96 < N; t += 128) {
      uint4 w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = ur[(size_t)(t + 32 * i) * (kD / 8)];
#pragma unroll
      for (int i = 0; i < 4; ++i) add_row(w[i]);
    }
    for (; t < N; t += 32) add_row(ur[(size_t)t * (kD / 8)]);
    float* part = reinterpret_cast<float*>(smem + SM::KQ);  // [32][kD]
#pragma unroll
    for (int y = 0; y < 8; ++y) part[p * kD + 8 * g + y] = su[y];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;
  const uint32_t tl = tm + ((uint32_t)(32 * (warp & 3)) << 16);  // this warp's lane quadrant
  if (tid < kD) {
    const float* part = reinterpret_cast<const float*>(smem + SM::KQ);
    float su = 0.0f;
#pragma unroll 8
    for (int p = 0; p < kTcThreads / 8; ++p) su += part[p * kD + tid];
    red[tid] = __fmaf_rn(etau, a.mu[(size_t)h * kD + tid], su);
  }
  __syncthreads();
  const float den = __fmul_rn(__fadd_rn(etau, (float)N), __fsqrt_rn((float)kD));
  // logit of token t: s = -(u_t . n) / ((e^tau + N) sqrt d)
  auto logit = [&](int t) -> float {
    const uint4* row = reinterpret_cast<const uint4*>(u + (size_t)t * kD);
    float dot = 0.0f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 w = row[c];
      const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        float lo, hi;
        unpack_bf16x2(wv[y], lo, hi);
        dot = __fmaf_rn(lo, red[8 * c + 2 * y], dot);
        dot = __fmaf_rn(hi, red[8 * c + 2 * y + 1], dot);
      }
    }
    return -__fdiv_rn(dot, den);
  };
  // ---- maximum logit m, P and E~ = sum e^{s - m} in one pass (thread per token): each thread
  //      keeps its exponential sum relative to its own running maximum, and the partial sums
  //      are rescaled to the common maximum when they are combined ----
  const bool keep = N <= SM::kSlogMax;
  float lmax = -INFINITY, lsum = 0.0f, lexp = 0.0f;
  for (int t = tid; t < N; t += kTcThreads) {
    const float s = logit(t);
    if (keep) slog[t] = s;
    const float mn = fmaxf(lmax, s);
    lexp = __fmaf_rn(lexp, expf(__fsub_rn(lmax, mn)), expf(__fsub_rn(s, mn)));
    lmax = mn;
    lsum += s;
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, lmax, o);
    const float oe = __shfl_xor_sync(0xffffffffu, lexp, o);
    const float mn = fmaxf(lmax, om);
    lexp = mn == -INFINITY ? 0.0f
                           : __fmaf_rn(lexp, expf(__fsub_rn(lmax, mn)), oe * expf(__fsub_rn(om, mn)));
    lmax = mn;
    lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
  }
  if ((tid & 31) == 0) {
    red[kD + warp] = lmax;
    red[kD + 8 + warp] = lsum;
    red[kD + 16 + warp] = lexp;
  }
  __syncthreads();
  float m = -INFINITY, P = 0.0f;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    m = fmaxf(m, red[kD + w]);
    P += red[kD + 8 + w];
  }
  if (!isfinite(m)) report(a.status, kErrRange);
  float Et = 0.0f;
#pragma unroll
  for (int w = 0; w < 8; ++w) Et += red[kD + 16 + w] * expf(__fsub_rn(red[kD + w], m));

  // ---- states over the token tiles ----
  constexpr uint32_t id_st = idesc_bf16_f32(128, kD, true, true);
  const uint32_t base = smem_u32(smem);
  const int NT = (N + kTcT - 1) / kTcT;
  auto pc = [hf](int c) { return pair_chunk(hf, c); };
  uint32_t phase = 0;
  bool ok = true;
  for (int tt = 0; tt < NT && ok; ++tt) {
    const int t = tt * kTcT + r;
    const bool valid = t < N;
    float x[32];
    unpack_half(kw, x);
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) ss = __fmaf_rn(x[i], x[i], ss);
    nrm[hf * kTcT + r] = ss;
    __syncthreads();
    unit_rot_half(a, t, valid, hf, nrm[r] + nrm[kTcT + r], x);
    put_half_pairs(smem + SM::KQ, r, hf, x);
    unpack_half(vw, x);
    put_half_pairs(smem + SM::AV, r, hf, x);
    const float s = valid ? (keep ? slog[t] : logit(t)) : 0.0f;
    const float e = valid ? expf(__fsub_rn(s, m)) : 0.0f;
    put_split(smem + SM::EVH, smem + SM::EVL, r, e, x, pc);
    put_split(smem + SM::SVH, smem + SM::SVL, r, s, x, pc);
    fence_proxy_async_smem();
    __syncthreads();
    {  // the next tile's k and v (or the first q tile's words, after the last state tile)
      const int tn = t + kTcT;
      if (tt + 1 < NT) {
        load_half_pairs(k + (size_t)tn * kD, tn < N, hf, kw);
        load_half_pairs(v + (size_t)tn * kD, tn < N, hf, vw);
      } else {
        load_half_pairs(q + (size_t)r * kD, r < N, hf, kw);
      }
    }
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kTcT / 16; ++kk) {
        const uint32_t off = kk * 2048;  // 16 token rows per step
        const uint32_t acc = (tt > 0 || kk > 0) ? 1u : 0u;
        const uint64_t bk = sw128_desc(base + SM::KQ + off, kAtom, 1024);
        mma_f16kind(tm, sw128_desc(base + SM::EVH + off, kAtom, 1024), bk, id_st, acc);
        mma_f16kind(tm, sw128_desc(base + SM::EVL + off, kAtom, 1024), bk, id_st, 1u);
        mma_f16kind(tm + 64, sw128_desc(base + SM::AV + off, kAtom, 1024), bk, id_st, acc);
      }
      mma_commit(bar);
    }
    ok = mbar_wait(bar, phase, abort_flag);
    phase ^= 1u;
    tc_fence_after();
    ok = __syncthreads_and(ok) != 0;  // uniform, and the tiles may be rewritten
  }
  if (!ok) report(a.status, kErrTimeout);

  // ---- states -> K-major bf16 hi/lo tiles: rows 0..63 F~, 64..127 G (D1), 128..191 H (D2);
  //      this thread copies key columns 32 hf .. 32 hf + 31 of its lane's rows ----
  if (ok) {
    auto cc = [hf](int c) { return 4 * hf + c; };
    float x[32];
    tmem_ld32(tl + 32 * hf, x);
    put_split(smem + SM::BHI, smem + SM::BLO, r, 1.0f, x, cc);
    if ((warp & 3) < 2) {  // lanes 0..63 of D2 (warp-uniform)
      tmem_ld32(tl + 64 + 32 * hf, x);
      put_split(smem + SM::BHI, smem + SM::BLO, 128 + r, 1.0f, x, cc);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- outputs per token tile: D3 = Q_hat [F~|G|H], combined with the row coefficients; this
  //      thread writes output columns 32 hf .. 32 hf + 31 of its row ----
  constexpr uint32_t id_out = idesc_bf16_f32(128, 3 * kD, false, false);
  const float rN = __fdiv_rn(1.0f, (float)N);
  for (int tt = 0; tt < NT && ok; ++tt) {
    const int t = tt * kTcT + r;
    const bool valid = t < N;
    float x[32];
    unpack_half(kw, x);  // this tile's q words
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) ss = __fmaf_rn(x[i], x[i], ss);
    nrm[hf * kTcT + r] = ss;
    __syncthreads();
    unit_rot_half(a, t, valid, hf, nrm[r] + nrm[kTcT + r], x);
    put_half_pairs(smem + SM::KQ, r, hf, x);
    float al = 0.0f, be = 0.0f, ga = 0.0f;
    if (valid) {
      const size_t row = row0 + t;
      const float sig1 = sigmoid(a.g1[row]), sigh = sigmoid(a.gh[row]);
      be = __fmul_rn(__fsub_rn(sig1, sigh), rN);
      ga = -__fadd_rn(__fmul_rn(__fmul_rn(be, P), rN), __fmul_rn(sigh, rN));
      if (a.g0) ga = __fadd_rn(ga, __fmul_rn(sigmoid(a.g0[row]), rN));
      al = __fdiv_rn(sigh, Et);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tt + 1 < NT) {  // the next tile's q words, while this tile's product runs
      const int tn = t + kTcT;
      load_half_pairs(q + (size_t)tn * kD, tn < N, hf, kw);
    }
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        const uint32_t off = kk * 32;  // 16 K values = 32 bytes inside the swizzled row
        const uint64_t aq = sw128_desc(base + SM::KQ + off, 16, 1024);
        mma_f16kind(tm, aq, sw128_desc(base + SM::BHI + off, 16, 1024), id_out, kk > 0 ? 1u : 0u);
        mma_f16kind(tm, aq, sw128_desc(base + SM::BLO + off, 16, 1024), id_out, 1u);
      }
      mma_commit(bar);
    }
    ok = mbar_wait(bar, phase, abort_flag);
    phase ^= 1u;
    tc_fence_after();
    ok = __syncthreads_and(ok) != 0;  // uniform before the aligned TMEM loads
    if (!ok) break;
    float o[32];
    {
      float f[32], g2[32], hh[32];
      tmem_ld32(tl + 32 * hf, f);
      tmem_ld32(tl + 64 + 32 * hf, g2);
      tmem_ld32(tl + 128 + 32 * hf, hh);
#pragma unroll
      for (int j = 0; j < 32; ++j)
        o[j] = __fmaf_rn(al, f[j], __fmaf_rn(be, g2[j], __fmul_rn(ga, hh[j])));
    }
    if (a.ln) {
      // output LayerNorm over the row: each half's mean and M2 over its 32 columns, merged
      // with the other half's (pairwise update for equal counts, half 0 first)
      float mean = 0.0f;
#pragma unroll
      for (int j = 0; j < 32; ++j) mean += o[j];
      mean *= (1.0f / 32.0f);
      float m2 = 0.0f;
#pragma unroll
      for (int j = 0; j < 32; ++j) m2 = __fmaf_rn(o[j] - mean, o[j] - mean, m2);
      lnx[hf * kTcT + r] = make_float2(mean, m2);
      __syncthreads();
      const float2 h0 = lnx[r], h1 = lnx[kTcT + r];
      const float dlt = h1.x - h0.x;
      const float mu_r = 0.5f * (h0.x + h1.x);
      const float var = (h0.y + h1.y + dlt * dlt * 16.0f) * (1.0f / kD);
      const float rstd = rsqrtf(var + a.ln_eps);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int col = 32 * hf + j;
        const float w = a.ln_w ? a.ln_w[(size_t)h * kD + col] : 1.0f;
        const float b = a.ln_b ? a.ln_b[(size_t)h * kD + col] : 0.0f;
        o[j] = __fmaf_rn((o[j] - mu_r) * rstd, w, b);
      }
    }
    {
      // the row's 64 output bytes as four 16-byte chunks, transposed within each group of four
      // lanes (rows 4g .. 4g + 3 of the warp) so that each store instruction writes whole 64-byte
      // row segments of eight rows: afterwards lane 4g + j holds chunk j of the row 4g + k in x[k]
      uint4 x[4];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        x[c] = make_uint4(pack_bf16x2(o[8 * c], o[8 * c + 1]), pack_bf16x2(o[8 * c + 2], o[8 * c + 3]),
                          pack_bf16x2(o[8 * c + 4], o[8 * c + 5]),
                          pack_bf16x2(o[8 * c + 6], o[8 * c + 7]));
      const int lane = tid & 31, j = lane & 3;
#pragma unroll
      for (int m = 1; m <= 2; m <<= 1) {
        const bool up = (j & m) != 0;
#pragma unroll
        for (int s0 = 0; s0 < 4; ++s0) {
          if (s0 & m) continue;  // the pair (s0, s0 | m)
          const uint4 send = up ? x[s0] : x[s0 | m];
          uint4 recv;
          recv.x = __shfl_xor_sync(0xffffffffu, send.x, m);
          recv.y = __shfl_xor_sync(0xffffffffu, send.y, m);
          recv.z = __shfl_xor_sync(0xffffffffu, send.z, m);
          recv.w = __shfl_xor_sync(0xffffffffu, send.w, m);
          if (up)
            x[s0] = recv;
          else
            x[s0 | m] = recv;
        }
      }
      const int t4 = t - (lane & 3);  // token of the group's first row
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (t4 + k < N)
          reinterpret_cast<uint4*>(out + (size_t)(t4 + k) * kD)[4 * hf + j] = x[k];
    }
    tc_fence_before();
    __syncthreads();  // D3 read and the q tile consumed before the next tile
  }
  if (!ok) {
    report(a.status, kErrTimeout);
    // the products of the phase that was not observed must finish before TMEM is released
    if (tid == 0) {
      int never = 0;
      mbar_wait(bar, phase ^ 1u, &never, 1ll << 32);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tm, 256);
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
  if (!f32 && a.N <= kTcNMax) {  // bf16: both contractions on the tensor cores
    static std::atomic<uint64_t> tc_set{0};
    if (!(tc_set.load() & bit)) {
      e = cudaFuncSetAttribute(enc_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)EncTcSmem::BYTES);
      if (e != cudaSuccess) return e;
      tc_set.fetch_or(bit);
    }
    enc_tc_kernel<<<a.B * a.H, kTcThreads, EncTcSmem::BYTES, stream>>>(a);
  } else if (f32) {
    enc_kernel<float><<<a.B * a.H, kNT, EncSmem::BYTES, stream>>>(a);
  } else {
    enc_kernel<__nv_bfloat16><<<a.B * a.H, kNT, EncSmem::BYTES, stream>>>(a);
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace zs
