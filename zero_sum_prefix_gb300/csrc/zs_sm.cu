// ZeroS-SM: the zero-sum reweighting applied to standard softmax attention (the quadratic
// variant).  Paper-Notes "ZeroS: Zero-Sum Linear Attention for Efficient Transformers", method
// details / linear-time prefix scan ("the same reweighting can be applied to standard softmax
// attention"), experiments (ZeroS-SM rows of the MAD and WikiText-103 tables).  The pages do not
// print its formula; the reading implemented here: logits s_{t,i} = q_t k_i^T / sqrt d (rotary
// positions when asked), and per query t over its keys i (i <= t, or every key in encoder mode,
// where t := N):
//   w_{t,i} = sig1_t delta_{t,i}/t + sigh_t eps_{t,i} (+ sig0_t/t),
//   delta_{t,i} = s_{t,i} - P_t/t,  eps_{t,i} = e^{s_{t,i}}/E_t - 1/t - delta_{t,i}/t,
// with P_t = sum_i s_{t,i} and E_t = sum_i e^{s_{t,i}}.  Expanding,
//   w_{t,i} = alpha_t e^{s_{t,i} - m_t} + beta_t s_{t,i} + gamma_t,
//   alpha_t = sigh_t / (E_t e^{-m_t}),  beta_t = (sig1_t - sigh_t)/t,
//   gamma_t = -beta_t P_t/t - sigh_t/t (+ sig0_t/t),                 o_t = sum_i w_{t,i} v_i.
//
// Kernel (one CTA per 128-query tile of one (b, h), heaviest causal tiles first): two passes
// over the key tiles.  Pass 1 computes S = Q K^T on the tensor cores (tcgen05.mma, accumulator
// in TMEM) and, per query row, the running maximum, the scaled exp-sum and the logit sum.  Pass 2
// recomputes S, forms W in fp32 from the final row statistics (the three terms nearly cancel,
// since the weights sum to zero, so W is rounded to bf16 only once, as a whole), writes it to
// TMEM and accumulates O += W V with W as the TMEM A operand.  Two epilogue warpgroups take the
// even and odd key tiles (two S buffers, two W buffers), so the exponentials of one tile overlap
// the other's; the row statistics of the two halves are merged between the passes.
//
// Warps: 0 = TMA producer (Q once; K per pass-1 tile; K and V per pass-2 tile, through a ring
// of stages), 1 = TMEM allocation and the single MMA-issuing thread, 4-7 and 8-11 = epilogue
// warpgroups (TMEM lane quadrant = warp % 4, one query row per thread).  Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include <algorithm>
#include <atomic>

#include "zs_common.cuh"
#include "zs_internal.h"
#include "zs_sm100.cuh"

namespace zs {
namespace {

using namespace sm100;

constexpr int kT = 128;                  // query rows per CTA, keys per tile
constexpr int kSmThreads = 384;          // 12 warps
constexpr uint32_t kAtom = 128 * 128;    // one [128 x 64] bf16 tile, 128-byte swizzle

template <int D>
struct SmCfg {
  static constexpr int KA = D / 64;                        // atom tiles along d
  static constexpr int NS = (D == 64) ? 4 : 3;             // K/V stages
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t STAGE_OFF = Q_OFF + KA * kAtom;
  static constexpr uint32_t STAGE = 2 * KA * kAtom;        // K then V
  static constexpr uint32_t STAT_OFF = STAGE_OFF + NS * STAGE;  // float4 [128] row stats
  static constexpr uint32_t MISC_OFF = STAT_OFF + kT * 16;
  static constexpr uint32_t BYTES = MISC_OFF + 256;
  static_assert(BYTES <= 232448, "shared memory budget of one CTA");
  // TMEM columns: S buffers, output accumulator, W buffers (bf16 pairs)
  static constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O = 256, TM_W0 = 384, TM_W1 = 448;
};

struct SmMisc {
  uint64_t q_full;
  uint64_t kv_full[4], kv_empty[4];
  uint64_t s_full[2], s_free[2], w_full[2], w_free[2];
  uint64_t o_full, fin;
  uint32_t tmem;
  int abort;
  int never;
};
static_assert(sizeof(SmMisc) <= 256, "SmMisc fits its slot");

struct SmParams {
  CUtensorMap tq, tk, tv;  // [B*H, N, d] bf16, box {64, 128, 1}, 128-byte swizzle
  SmArgs a;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Number of key tiles a query tile visits and the key count t of each row.
__device__ __forceinline__ int key_tiles(const SmArgs& a, int qt) {
  return a.causal ? qt + 1 : (a.N + kT - 1) / kT;
}

// Index of pass-2 item g among the pass-2 items of the same buffer (g & 1); J = key tiles.
__device__ __forceinline__ int p2_index(int g, int J) {
  const int first = J + ((J ^ g) & 1);
  return (g - first) >> 1;
}

// ------------------------------------------------------------------------------ producer
template <int D>
__device__ void sm_producer(const SmParams& p, uint8_t* smem, SmMisc* ms, int bh, int qt, int J) {
  using CF = SmCfg<D>;
  const uint32_t base = smem_u32(smem);
  mbar_arrive_expect_tx(&ms->q_full, CF::KA * kAtom);
#pragma unroll
  for (int at = 0; at < CF::KA; ++at)
    tma_load_3d(base + CF::Q_OFF + at * kAtom, &p.tq, 64 * at, qt * kT, bh, &ms->q_full);
  for (int g = 0; g < 2 * J; ++g) {
    const int st = g % CF::NS;
    if (g >= CF::NS && !mbar_wait(&ms->kv_empty[st], ((g / CF::NS) - 1) & 1, &ms->abort)) {
      report(p.a.status, kErrTimeout);
      ms->abort = 1;
      return;
    }
    const bool pass2 = g >= J;
    const int j = pass2 ? g - J : g;
    const uint32_t kt = base + CF::STAGE_OFF + st * CF::STAGE;
    mbar_arrive_expect_tx(&ms->kv_full[st], (pass2 ? 2 : 1) * CF::KA * kAtom);
#pragma unroll
    for (int at = 0; at < CF::KA; ++at)
      tma_load_3d(kt + at * kAtom, &p.tk, 64 * at, j * kT, bh, &ms->kv_full[st]);
    if (pass2) {
#pragma unroll
      for (int at = 0; at < CF::KA; ++at)
        tma_load_3d(kt + (CF::KA + at) * kAtom, &p.tv, 64 * at, j * kT, bh, &ms->kv_full[st]);
    }
  }
}

// ------------------------------------------------------------------------------ MMA issuer
template <int D>
__device__ void sm_mma(const SmArgs& a, uint8_t* smem, SmMisc* ms, int J) {
  using CF = SmCfg<D>;
  const uint32_t base = smem_u32(smem);
  const uint32_t tm = ms->tmem;
  constexpr uint32_t id_qk = idesc_bf16_f32(128, 128, false, false);  // S = Q K^T
  constexpr uint32_t id_ov = idesc_bf16_f32(128, D, false, true);      // O += W V
  // O += W V for the pass-2 item g (W from TMEM, V MN-major in its stage)
  auto issue_wv = [&](int g) -> bool {
    const int b = g & 1, j = g - J;
    if (!mbar_wait(&ms->w_full[b], p2_index(g, J) & 1, &ms->abort)) return false;
    tc_fence_after();
    const uint32_t vt = base + CF::STAGE_OFF + (g % CF::NS) * CF::STAGE + CF::KA * kAtom;
    const uint32_t tw = tm + (b ? CF::TM_W1 : CF::TM_W0);
#pragma unroll
    for (int kk = 0; kk < kT / 16; ++kk)
      mma_f16kind_ts(tm + CF::TM_O, tw + kk * 8, sw128_desc(vt + kk * 2048, kAtom, 1024), id_ov,
                  (j > 0 || kk > 0) ? 1u : 0u);
    mma_commit(&ms->w_free[b]);
    mma_commit(&ms->kv_empty[g % CF::NS]);
    return true;
  };
  bool ok = mbar_wait(&ms->q_full, 0, &ms->abort);
  for (int g = 0; g < 2 * J && ok; ++g) {
    const int st = g % CF::NS, b = g & 1;
    ok = mbar_wait(&ms->kv_full[st], (g / CF::NS) & 1, &ms->abort);
    if (ok && g >= 2) ok = mbar_wait(&ms->s_free[b], ((g >> 1) - 1) & 1, &ms->abort);
    if (!ok) break;
    tc_fence_after();
    const uint32_t qs = base + CF::Q_OFF, ks = base + CF::STAGE_OFF + st * CF::STAGE;
    const uint32_t ts = tm + (b ? CF::TM_S1 : CF::TM_S0);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk / 4) * kAtom + (kk % 4) * 32;
      mma_f16kind(ts, sw128_desc(qs + off, 16, 1024), sw128_desc(ks + off, 16, 1024), id_qk,
               kk > 0 ? 1u : 0u);
    }
    mma_commit(&ms->s_full[b]);
    if (g < J) mma_commit(&ms->kv_empty[st]);  // pass 1 reads K only
    if (g >= J + 1) ok = issue_wv(g - 1);      // the previous tile's W is due by now
  }
  if (ok && J > 0) ok = issue_wv(2 * J - 1);
  if (ok) mma_commit(&ms->o_full);
  if (!ok) {
    report(a.status, kErrTimeout);
    ms->abort = 1;
  }
  mma_commit(&ms->fin);
}

// ------------------------------------------------------------------------------ epilogue
// Warpgroup w (0 or 1) handles the key tiles of parity w in both passes; thread = query row.
template <int D>
__device__ void sm_epilogue(const SmArgs& a, uint8_t* smem, SmMisc* ms, int bh, int qt, int J,
                            int w) {
  using CF = SmCfg<D>;
  const int wq = (threadIdx.x >> 5) & 3;
  const int r = wq * 32 + (threadIdx.x & 31);
  const uint32_t tl = ms->tmem + ((uint32_t)(wq * 32) << 16);
  const uint32_t ts = tl + (w ? CF::TM_S1 : CF::TM_S0);
  const uint32_t tw = tl + (w ? CF::TM_W1 : CF::TM_W0);
  const int t = qt * kT + r;                      // query index (0-based)
  const bool row_ok = t < a.N;
  const size_t row = (size_t)bh * a.N + t;
  const int lim = a.causal ? t : a.N - 1;         // last key of this query
  // last key visible to every row of this warp: a tile is unmasked for the whole warp when it
  // ends at or before it (uniform across the warp, as the .sync.aligned TMEM loads require)
  const int lim_warp = a.causal ? qt * kT + wq * 32 : a.N - 1;
  const float tc = a.causal ? (float)(t + 1) : (float)a.N;
  const float inv_sqrt_d = 1.0f / sqrtf((float)D);
  const float c2 = 1.4426950408889634f * inv_sqrt_d;  // log2(e) / sqrt(d): exponent in base 2
  bool ok = true;

  // ---- pass 1: running maximum (base-2 units), scaled exp-sum and logit sum ----
  float m2 = -INFINITY, l = 0.0f, P = 0.0f;
  for (int g = w; g < J && ok; g += 2) {
    ok = mbar_wait_warp(&ms->s_full[w], (g >> 1) & 1, &ms->abort);
    if (!ok) break;
    tc_fence_after();
    const int k0 = g * kT;
    const bool full = k0 + kT - 1 <= lim_warp;
    if (full) {  // every key visible: packed fp32 arithmetic, loads double-buffered
      uint32_t ra[32], rb[32];
      auto stat_chunk = [&](uint32_t (&rv)[32]) {
        float cm = __uint_as_float(rv[0]);
        float2 ps = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int y = 0; y < 16; ++y) {
          const float2 xv = make_float2(__uint_as_float(rv[2 * y]), __uint_as_float(rv[2 * y + 1]));
          cm = fmaxf(cm, fmaxf(xv.x, xv.y));
          ps = __fadd2_rn(ps, xv);
        }
        const float mn = fmaxf(m2, cm * c2);
        const float2 c2v = make_float2(c2, c2), nm = make_float2(-mn, -mn);
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int y = 0; y < 16; ++y) {
          const float2 e = __ffma2_rn(
              make_float2(__uint_as_float(rv[2 * y]), __uint_as_float(rv[2 * y + 1])), c2v, nm);
          acc = __fadd2_rn(acc, make_float2(ex2(e.x), ex2(e.y)));
        }
        l = fmaf(l, ex2(m2 - mn), acc.x + acc.y);
        m2 = mn;
        P += ps.x + ps.y;
      };
      tmem_ld32_nowait(ts, ra);
      tmem_wait_ld();
      reg_fence(ra);
      tmem_ld32_nowait(ts + 32, rb);
      stat_chunk(ra);
      tmem_wait_ld();
      reg_fence(rb);
      tmem_ld32_nowait(ts + 64, ra);
      stat_chunk(rb);
      tmem_wait_ld();
      reg_fence(ra);
      tmem_ld32_nowait(ts + 96, rb);
      stat_chunk(ra);
      tmem_wait_ld();
      reg_fence(rb);
      tc_fence_before();
      mbar_arrive(&ms->s_free[w]);  // every column of S is in registers: release the buffer
      stat_chunk(rb);
      continue;
    }
#pragma unroll 1
    for (int ch = 0; ch < 4; ++ch) {
      float v[32];
      __syncwarp();  // the rows of a warp diverge below; the TMEM load needs all 32 lanes
      tmem_ld32(ts + 32 * ch, v);
      float cm = -INFINITY, cs = 0.0f;
#pragma unroll
      for (int x = 0; x < 32; ++x) {
        const bool valid = full || k0 + 32 * ch + x <= lim;
        if (valid) {
          cm = fmaxf(cm, v[x]);
          cs += v[x];
        }
      }
      if (cm == -INFINITY) continue;  // no key of this chunk is visible to the row
      const float mn = fmaxf(m2, cm * c2);
      float acc = 0.0f;
#pragma unroll
      for (int x = 0; x < 32; ++x) {
        const bool valid = full || k0 + 32 * ch + x <= lim;
        if (valid) acc += ex2(fmaf(v[x], c2, -mn));
      }
      l = fmaf(l, ex2(m2 - mn), acc);
      m2 = mn;
      P += cs;
    }
    tc_fence_before();
    mbar_arrive(&ms->s_free[w]);
  }
  if (!ok) ms->abort = 1;
  // ---- merge the two halves' statistics: warpgroup 0 publishes its row's, warpgroup 1
  // merges and publishes the result (both warpgroups reach both barriers) ----
  float4* stat = reinterpret_cast<float4*>(smem + CF::STAT_OFF);
  if (w == 0) stat[r] = make_float4(m2, l, P, 0.0f);
  named_bar_sync(1, 256);
  if (w == 1) {
    const float4 o = stat[r];
    if (o.x != -INFINITY) {
      const float mn = fmaxf(m2, o.x);
      l = l * ex2(m2 - mn) + o.y * ex2(o.x - mn);
      m2 = mn;
    }
    P += o.z;
    stat[r] = make_float4(m2, l, P, 0.0f);
  }
  named_bar_sync(1, 256);
  if (w == 0) {
    const float4 o = stat[r];
    m2 = o.x;
    l = o.y;
    P = o.z;
  }
  if (ms->abort) return;

  // ---- coefficients of the row: w = alpha 2^{c2 raw - m2} + bs raw + gamma ----
  float sig1 = 0.0f, sigh = 0.0f, sig0 = 0.0f;
  if (row_ok) {
    sig1 = sigmoid(a.g1[row]);
    sigh = sigmoid(a.gh[row]);
    if (a.g0) sig0 = sigmoid(a.g0[row]);
  }
  const float rt = 1.0f / tc;
  const float alpha = sigh / l;
  const float beta = (sig1 - sigh) * rt;
  const float bs = beta * inv_sqrt_d;
  const float gamma = fmaf(-beta * P * inv_sqrt_d, rt, (sig0 - sigh) * rt);

  // ---- pass 2: W tiles (bf16, rounded once) for the O += W V products ----
  for (int g = J + ((J ^ w) & 1); g < 2 * J && ok; g += 2) {
    const int n = p2_index(g, J), j = g - J;
    ok = mbar_wait_warp(&ms->s_full[w], (g >> 1) & 1, &ms->abort);
    if (ok && n >= 1) ok = mbar_wait_warp(&ms->w_free[w], (n - 1) & 1, &ms->abort);
    if (!ok) break;
    tc_fence_after();
    const int k0 = j * kT;
    const bool full = k0 + kT - 1 <= lim_warp;
    if (full) {  // every key visible: packed fp32 arithmetic, loads double-buffered
      const float2 c2v = make_float2(c2, c2), nm = make_float2(-m2, -m2);
      const float2 av = make_float2(alpha, alpha), bv = make_float2(bs, bs);
      const float2 gv = make_float2(gamma, gamma);
      uint32_t ra[32], rb[32];
      auto w_chunk = [&](uint32_t (&rv)[32], int ch) {
        uint32_t pk[16];
#pragma unroll
        for (int y = 0; y < 16; ++y) {
          const float2 xv = make_float2(__uint_as_float(rv[2 * y]), __uint_as_float(rv[2 * y + 1]));
          float2 e = __ffma2_rn(xv, c2v, nm);
          e = make_float2(ex2(e.x), ex2(e.y));
          const float2 wv = __ffma2_rn(e, av, __ffma2_rn(xv, bv, gv));
          pk[y] = pack_bf16x2(wv.x, wv.y);
        }
        tmem_st16_nowait(tw + 16 * ch, pk);
      };
      tmem_ld32_nowait(ts, ra);
      tmem_wait_ld();
      reg_fence(ra);
      tmem_ld32_nowait(ts + 32, rb);
      w_chunk(ra, 0);
      tmem_wait_ld();
      reg_fence(rb);
      tmem_ld32_nowait(ts + 64, ra);
      w_chunk(rb, 1);
      tmem_wait_ld();
      reg_fence(ra);
      tmem_ld32_nowait(ts + 96, rb);
      w_chunk(ra, 2);
      tmem_wait_ld();
      reg_fence(rb);
      tc_fence_before();
      mbar_arrive(&ms->s_free[w]);  // every column of S is in registers: release the buffer
      w_chunk(rb, 3);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&ms->w_full[w]);
      continue;
    }
#pragma unroll 1
    for (int ch = 0; ch < 4; ++ch) {
      float v[32];
      __syncwarp();
      tmem_ld32(ts + 32 * ch, v);
      uint32_t pk[16];
#pragma unroll
      for (int y = 0; y < 16; ++y) {
        float wv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int x = 2 * y + e;
          const bool valid = full || k0 + 32 * ch + x <= lim;
          wv[e] = valid ? fmaf(alpha, ex2(fmaf(v[x], c2, -m2)), fmaf(bs, v[x], gamma)) : 0.0f;
        }
        pk[y] = pack_bf16x2(wv[0], wv[1]);
      }
      tmem_st16_nowait(tw + 16 * ch, pk);
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&ms->s_free[w]);
    mbar_arrive(&ms->w_full[w]);
  }
  if (!ok) {
    report(a.status, kErrTimeout);
    ms->abort = 1;
    return;
  }
  // ---- output: warpgroup w writes columns [w D/2, (w + 1) D/2) of its rows ----
  if (!mbar_wait_warp(&ms->o_full, 0, &ms->abort)) {
    report(a.status, kErrTimeout);
    ms->abort = 1;
    return;
  }
  tc_fence_after();
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
#pragma unroll
  for (int cb = 0; cb < D / 64; ++cb) {
    const int c0 = w * (D / 2) + 32 * cb;
    float v[32];
    tmem_ld32(tl + CF::TM_O + c0, v);
    if (row_ok) {
      uint4* dst = reinterpret_cast<uint4*>(out + row * D + c0);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        dst[q4] = make_uint4(pack_bf16x2(v[8 * q4 + 0], v[8 * q4 + 1]),
                             pack_bf16x2(v[8 * q4 + 2], v[8 * q4 + 3]),
                             pack_bf16x2(v[8 * q4 + 4], v[8 * q4 + 5]),
                             pack_bf16x2(v[8 * q4 + 6], v[8 * q4 + 7]));
    }
  }
}

// ============================================================================ kernel
template <int D>
__global__ void __launch_bounds__(kSmThreads, 1) sm_kernel(const __grid_constant__ SmParams p) {
  using CF = SmCfg<D>;
  const SmArgs& a = p.a;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (smem_u32(smem) & 1023u) {  // the swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) report(a.status, kErrUnsupported);
    return;
  }
  SmMisc* ms = reinterpret_cast<SmMisc*>(smem + CF::MISC_OFF);
  const int warp = threadIdx.x >> 5;
  const int nqt = (a.N + kT - 1) / kT;
  // every sequence's heaviest (last) causal query tile first, then the next lighter ones
  const int qt = a.causal ? nqt - 1 - (int)blockIdx.y : (int)blockIdx.y;
  const int bh = blockIdx.x;
  const int J = key_tiles(a, qt);
  if (threadIdx.x == 0) {
    mbar_init(&ms->q_full, 1);
    for (int i = 0; i < CF::NS; ++i) {
      mbar_init(&ms->kv_full[i], 1);
      mbar_init(&ms->kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms->s_full[i], 1);
      mbar_init(&ms->s_free[i], 128);
      mbar_init(&ms->w_full[i], 128);
      mbar_init(&ms->w_free[i], 1);
    }
    mbar_init(&ms->o_full, 1);
    mbar_init(&ms->fin, 1);
    ms->abort = 0;
    ms->never = 0;
  }
  if (warp == 1) {
    tmem_alloc(&ms->tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 0) {
    if ((threadIdx.x & 31) == 0) sm_producer<D>(p, smem, ms, bh, qt, J);
  } else if (warp == 1) {
    if ((threadIdx.x & 31) == 0) sm_mma<D>(a, smem, ms, J);
  } else if (warp >= 4) {
    sm_epilogue<D>(a, smem, ms, bh, qt, J, (warp - 4) >> 2);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    // every MMA has completed once `fin` fires (it is committed after the last one)
    if (!mbar_wait(&ms->fin, 0, &ms->never, 4000000000ull)) report(a.status, kErrTimeout);
    tc_fence_after();
    tmem_dealloc(ms->tmem, 512);
  }
}

// ============================================================================ one-pass, d = 64
// Expanding the weights per query row, o_t = alpha_t A_t + beta_t B_t + gamma_t C_t with
//   A_t = sum_i 2^{c2 x_{t,i} - m_t} v_i,   B_t = sum_i x_{t,i} v_i / sqrt d,   C_t = sum_i v_i
// (i over the row's keys, x the raw logit q k^T, c2 = log2(e) / sqrt d, m_t a reference in
// base-2 units), and alpha_t = sigh_t / l_t with l_t = sum_i 2^{c2 x - m}, beta_t and gamma_t as
// above with P_t = sum_i x_{t,i} / sqrt d.  So one pass over the key tiles suffices: S = Q K^T
// once per tile; P = 2^{c2 x - m} and x itself rounded to bf16 and written over S's own fp32
// columns (piece h of 16 keys: P in columns 16 h .. 16 h + 7, x in 16 h + 8 .. 16 h + 15); then
// A += P V and B += X V.  The logit sum P_t is q_t . (sum of the earlier tiles' keys) plus the
// sum of the last tile's bf16 logits, the very values that B sums there: for the rows of the
// first query tile (few keys) the weights alpha P + beta x / sqrt d + gamma then sum to sig0 up to
// the fp32 rounding of the sums (exactly zero output for a single visible key), and elsewhere the
// roundings only perturb each weight.  C does not depend on the query: it is the sum of the value
// column sums of the key tiles before the diagonal one, and the diagonal tile's prefix comes from
// one product with a lower-triangular ones tile at the end.  The per-tile column sums of k and v
// and each tile's largest key norm come from a pass that also applies the rotary map; the norm
// bounds the tile's logits: where c2 |q_t| max |k| cannot exceed the reference by more than
// kRaise, the tile's maximum is not needed at all.
// Three S buffers: S_{n+3} is formed as soon as tile n's products are issued, so the tensor
// cores, the exponentials of tile n+1 and the products of tile n overlap.  Both epilogue
// warpgroups work on every key tile, warpgroup w on its keys 64 w .. 64 w + 63; where the bound
// does not settle it, the row's tile maximum is exchanged between the two warps that hold the
// row (a 64-thread barrier), and the reference m rises (lazily: only when the tile maximum
// exceeds it by more than kRaise = 16, so P <= 2^16) before the tile's P is formed; A and the
// exp-sums are then rescaled (warpgroup 0 rescales A, once the previous tile's products have
// completed).
// Persistent: one CTA per SM takes the query tiles ("items", heaviest first) c, c + G, c + 2G, ...
// (G CTAs), and every role runs through one sequence of key tiles n counted over its items, so
// the next item's Q and K/V loads and its first S products overlap the current item's last
// products and output (the per-CTA start and drain are paid once per SM instead of once per
// query tile).  An item's C goes into its diagonal tile's own S buffer (the products of that tile
// have read it by then: the tensor-core operations of one thread run in order); the next item's
// third S product, which uses that buffer, waits until the output has read C, A and B.
// TMEM (512 columns): S0, S1, S2 (128 each), A (64), B (64).
struct Sm1Cfg {
  static constexpr int NS = 5;                             // K/V stages
  static constexpr int NB = 3;                             // S buffers
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t STAGE_OFF = Q_OFF + kAtom;
  static constexpr uint32_t STAGE = 2 * kAtom;             // K then V
  static constexpr uint32_t TRI_OFF = STAGE_OFF + NS * STAGE;  // [128 x 128] lower-triangular ones
  static constexpr uint32_t XMAX_OFF = TRI_OFF + 2 * kAtom;    // float [2 bufs][2 halves][128]
  static constexpr uint32_t STAT_OFF = XMAX_OFF + 4 * kT * 4;  // float2 [2][128] sums
  static constexpr uint32_t CBASE_OFF = STAT_OFF + 2 * kT * 8;  // float [2 items][64]
  // K_base, one copy per column-sum warp
  static constexpr uint32_t KBASE_OFF = CBASE_OFF + 2 * 64 * 4;  // float [2 items][2][64]
  // per row, by item parity: the gate logits (g1, gh, g0), q_t . K_base and the bound factor
  // c2 |q_t| (1 + slack)
  static constexpr uint32_t ROWV_OFF = KBASE_OFF + 2 * 2 * 64 * 4;  // float [2 items][5][128]
  static constexpr uint32_t MISC_OFF = ROWV_OFF + 2 * 5 * kT * 4;
  static constexpr uint32_t BYTES = MISC_OFF + 256;
  static_assert(BYTES <= 232448, "shared memory budget of one CTA");
  static constexpr uint32_t TM_A = 384, TM_B = 448;
  static constexpr float kRaise = 16.0f;  // base-2 units
  static constexpr float kBoundSlack = 1.001f;  // covers the fp32 rounding of logits and norms
};

__device__ __forceinline__ uint32_t sm1_sbuf(int i) { return 128u * (uint32_t)i; }

struct Sm1Misc {
  uint64_t q_full, q_empty;
  uint64_t kv_full[Sm1Cfg::NS], kv_empty[Sm1Cfg::NS];
  uint64_t s_full[3], w_full[3];
  uint64_t o_full, acc_free, fin;
  uint64_t cb_full[2], cb_empty[2];
  uint32_t tmem;
  int abort;
  int never;
};
static_assert(sizeof(Sm1Misc) <= 256, "Sm1Misc fits its slot");

// The query tile of work item i: every sequence's last causal query tile first, then the next
// lighter ones (in encoder mode all items have the same number of key tiles).
struct Sm1Item {
  int bh, qt, J;
};
__device__ __forceinline__ Sm1Item sm1_item(const SmArgs& a, int i) {
  const int BH = a.B * a.H, nqt = (a.N + kT - 1) / kT;
  const int y = i / BH;
  Sm1Item it;
  it.bh = i - y * BH;
  it.qt = a.causal ? nqt - 1 - y : y;
  it.J = key_tiles(a, it.qt);
  return it;
}
__device__ __forceinline__ int sm1_items(const SmArgs& a) {
  return a.B * a.H * ((a.N + kT - 1) / kT);
}
// The it-th item of this CTA: rounds of gridDim.x items, taken in alternating directions, so
// that every CTA's total of key tiles is about the same (items >= sm1_items when none is left).
__device__ __forceinline__ int sm1_mine(int it) {
  const int c = (it & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x;
  return it * (int)gridDim.x + c;
}


// Named barrier over nthreads threads that also returns whether any of them passed pred = true.
__device__ __forceinline__ bool named_bar_any(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0u;
}

// One lane: per item Q (once the previous item's Q has been read by its last S product and by
// the epilogue), then the item's K and V tiles through the stage ring.
__device__ void sm1_producer(const SmParams& p, uint8_t* smem, Sm1Misc* ms) {
  using CF = Sm1Cfg;
  const SmArgs& a = p.a;
  const uint32_t base = smem_u32(smem);
  const int nitems = sm1_items(a);
  int n = 0;  // key tiles loaded so far, over all items
  for (int it = 0, item = sm1_mine(0); item < nitems; item = sm1_mine(++it)) {
    const Sm1Item w = sm1_item(a, item);
    if (it >= 1 && !mbar_wait(&ms->q_empty, (it - 1) & 1, &ms->abort)) goto fail;
    mbar_arrive_expect_tx(&ms->q_full, kAtom);
    tma_load_3d(base + CF::Q_OFF, &p.tq, 0, w.qt * kT, w.bh, &ms->q_full);
    for (int g = 0; g < w.J; ++g, ++n) {
      const int st = n % CF::NS;
      if (n >= CF::NS && !mbar_wait(&ms->kv_empty[st], ((n / CF::NS) - 1) & 1, &ms->abort))
        goto fail;
      const uint32_t kt = base + CF::STAGE_OFF + st * CF::STAGE;
      mbar_arrive_expect_tx(&ms->kv_full[st], 2 * kAtom);
      tma_load_3d(kt, &p.tk, 0, g * kT, w.bh, &ms->kv_full[st]);
      tma_load_3d(kt + kAtom, &p.tv, 0, g * kT, w.bh, &ms->kv_full[st]);
    }
  }
  return;
fail:
  report(a.status, kErrTimeout);
  ms->abort = 1;
}

// Issue order per item: S of its first three key tiles (the third only once the previous item's
// output has read C, A and B: it uses the buffer that held C); then per key tile the products
// once both warpgroups have released it (A += P V, B += X V; the item's first products also wait
// until the previous item's A and B have been read), and S_{n+3} into the buffer those products
// have just read.  The tensor-core operations of one thread run in order, so S_{n+3} overwrites
// tile n's P and x only after its products have read them.  The whole warp runs this loop (its
// operands stay warp-uniform, so the issue stays short next to the busy epilogue warps of the
// same scheduler) and one elected lane issues; descriptors advance by plain additions (16 key
// rows of an MN-major tile = 2048 bytes = 128 units).
__device__ void sm1_mma(const SmArgs& a, uint8_t* smem, Sm1Misc* ms) {
  using CF = Sm1Cfg;
  const bool leader = elect_one();
  const uint32_t base = smem_u32(smem);
  const uint32_t tm = ms->tmem;
  const int nitems = sm1_items(a);
  constexpr uint32_t id_qk = idesc_bf16_f32(128, 128, false, false);  // S = Q K^T
  constexpr uint32_t id_pv = idesc_bf16_f32(128, 64, false, true);    // A += P V, B += X V
  const uint64_t qd = sw128_desc(base + CF::Q_OFF, 16, 1024);
  // S_n for key tile n (counted over all items) into buffer n % 3; after the item's last one, Q
  // is released (to the producer, once the epilogue has read it too)
  auto issue_s = [&](int n, bool last) -> bool {
    const int st = n % CF::NS;
    if (!mbar_wait_warp(&ms->kv_full[st], (n / CF::NS) & 1, &ms->abort)) return false;
    tc_fence_after();
    const uint64_t kd = sw128_desc(base + CF::STAGE_OFF + st * CF::STAGE, 16, 1024);
    const uint32_t ts = tm + sm1_sbuf(n % CF::NB);
    if (leader) {
      mma_f16kind(ts, qd, kd, id_qk, 0u);
#pragma unroll
      for (int kk = 1; kk < 4; ++kk) mma_f16kind(ts, qd + 2 * kk, kd + 2 * kk, id_qk, 1u);
      mma_commit(&ms->s_full[n % CF::NB]);
      if (last) mma_commit(&ms->q_empty);
    }
    __syncwarp();
    return true;
  };
  bool ok = true;
  int n0 = 0;  // the item's first key tile, counted over all items
  for (int it = 0, item = sm1_mine(0); ok && item < nitems; item = sm1_mine(++it)) {
    const int J = sm1_item(a, item).J;
    ok = mbar_wait_warp(&ms->q_full, it & 1, &ms->abort);
    for (int g = 0; g < CF::NB && g < J && ok; ++g) {
      if (g == CF::NB - 1 && it >= 1 && a.causal)
        ok = mbar_wait_warp(&ms->acc_free, (it - 1) & 1, &ms->abort);
      if (ok) ok = issue_s(n0 + g, g == J - 1);
    }
    for (int g = 0; g < J && ok; ++g) {
      const int n = n0 + g;
      const int b = n % CF::NB, st = n % CF::NS;
      const uint32_t vt = base + CF::STAGE_OFF + st * CF::STAGE + kAtom;
      const uint64_t vd = sw128_desc(vt, kAtom, 1024);
      const uint32_t ts = tm + sm1_sbuf(b);
      ok = mbar_wait_warp(&ms->w_full[b], (n / CF::NB) & 1, &ms->abort);
      if (ok && g == 0 && it >= 1) ok = mbar_wait_warp(&ms->acc_free, (it - 1) & 1, &ms->abort);
      if (!ok) break;
      tc_fence_after();
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk) {
          const uint32_t acc = (g > 0 || kk > 0) ? 1u : 0u;
          mma_f16kind_ts(tm + CF::TM_A, ts + 16 * kk, vd + 128 * kk, id_pv, acc);
          mma_f16kind_ts(tm + CF::TM_B, ts + 16 * kk + 8, vd + 128 * kk, id_pv, acc);
        }
        if (a.causal && g == J - 1) {
          // C of the diagonal tile: lower-triangular ones (K-major, two atoms of 64 keys) times
          // V, into this tile's own S buffer, after the products above have read it
          const uint64_t td = sw128_desc(base + CF::TRI_OFF, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            mma_f16kind(ts, td + (uint64_t)(((kk / 4) * kAtom + (kk % 4) * 32) >> 4),
                        vd + 128 * kk, id_pv, kk > 0 ? 1u : 0u);
        }
        mma_commit(&ms->kv_empty[st]);  // also tells the epilogue that A holds tile n
        if (g == J - 1) mma_commit(&ms->o_full);
      }
      __syncwarp();
      if (g + CF::NB < J) ok = issue_s(n + CF::NB, g + CF::NB == J - 1);
    }
    n0 += J;
  }
  if (leader) {
    if (!ok) {
      report(a.status, kErrTimeout);
      ms->abort = 1;
    }
    mma_commit(&ms->fin);
  }
  __syncwarp();
}

// Warps 2 and 3 (thread t = 0..63: C_base column t, query rows t and t + 64): per item the
// parts of C and P_t that are the same for every row, from the per-tile statistics: K_base = the
// key column sums of the tiles before the last one, C_base = the value column sums of the tiles
// before the diagonal one (all tiles in encoder mode); eight partial sums over the tiles
// (g = 8 j + u), added in a fixed order, so that the loads overlap; and the gate logits of the
// item's rows with the bound factor of their logits; once the query tile has landed, each row's
// q_t . K_base (each warp keeps its own copy of K_base).  Two buffers (by item parity): an
// item's values are written once the epilogue has used those of two items before, so their
// loads run ahead of the epilogue.
__device__ void sm1_colsum(const SmArgs& a, uint8_t* smem, Sm1Misc* ms) {
  using CF = Sm1Cfg;
  constexpr float c2 = 1.4426950408889634f * 0.125f;  // log2(e) / sqrt(d), d = 64
  const int t = threadIdx.x - 64;     // C_base column, and the rows t and t + 64
  const int c = t >> 5, l = t & 31;   // this warp (0, 1) and lane
  const int nt = (a.N + kT - 1) / kT;
  const int nitems = sm1_items(a);
  const uint32_t qrow = smem_u32(smem) + CF::Q_OFF;
  for (int it = 0, item = sm1_mine(0); item < nitems; item = sm1_mine(++it)) {
    const Sm1Item w = sm1_item(a, item);
    const int par = it & 1;
    if (it >= 2 && !mbar_wait_warp(&ms->cb_empty[par], ((it >> 1) - 1) & 1, &ms->abort)) {
      report(a.status, kErrTimeout);
      ms->abort = 1;
      return;
    }
    // K_base over all 64 columns (this lane: columns l and l + 32), C_base over the column t
    const float* st = a.kstat + (size_t)w.bh * nt * kSmStat;
    float pk0[8] = {}, pk1[8] = {}, pv[8] = {};
    const int nk = w.J - 1, nv = a.causal ? w.J - 1 : w.J;
    for (int g0 = 0; g0 < nv; g0 += 8) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int g = g0 + u;
        if (g < nk) {
          pk0[u] += st[(size_t)g * kSmStat + l];
          pk1[u] += st[(size_t)g * kSmStat + 32 + l];
        }
        if (g < nv) pv[u] += st[(size_t)g * kSmStat + 68 + t];
      }
    }
    auto sum8 = [](const float (&x)[8]) {
      return ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
    };
    float* kb = reinterpret_cast<float*>(smem + CF::KBASE_OFF) + (par * 2 + c) * 64;
    kb[l] = sum8(pk0);
    kb[32 + l] = sum8(pk1);
    reinterpret_cast<float*>(smem + CF::CBASE_OFF)[par * 64 + t] = sum8(pv);
    // per row rr (t and t + 64): the gate logits and the bound factor of its logits
    float* rowv = reinterpret_cast<float*>(smem + CF::ROWV_OFF) + par * 5 * kT;
    const float* qn = st + (size_t)w.qt * kSmStat + 132;  // the norms of the tile's q rows
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int rr = t + 64 * h, tq = w.qt * kT + rr;
      const bool valid = tq < a.N;
      const size_t row = (size_t)w.bh * a.N + tq;
      rowv[rr] = valid ? a.g1[row] : 0.0f;
      rowv[kT + rr] = valid ? a.gh[row] : 0.0f;
      rowv[2 * kT + rr] = (valid && a.g0) ? a.g0[row] : 0.0f;
      rowv[4 * kT + rr] = qn[rr] * (c2 * CF::kBoundSlack);
    }
    __syncwarp();
    // the earlier tiles' part of the logit sum of the rows t and t + 64, q_t . K_base (four
    // partial sums), once the query tile has landed; then Q is not read again here
    if (!mbar_wait_warp(&ms->q_full, par, &ms->abort)) {
      report(a.status, kErrTimeout);
      ms->abort = 1;
      return;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int rr = t + 64 * h;
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const uint4 u = lds128(qrow + sw128_off(rr, cc));
        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          float lo, hi;
          unpack_bf16x2(wv[y], lo, hi);
          acc[y] = __fmaf_rn(hi, kb[8 * cc + 2 * y + 1], __fmaf_rn(lo, kb[8 * cc + 2 * y], acc[y]));
        }
      }
      rowv[3 * kT + rr] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
    __syncwarp();
    if (l == 0) {
      mbar_arrive(&ms->cb_full[par]);  // count 2: both warps
      mbar_arrive(&ms->q_empty);       // count 3: the item's last S and both warps
    }
  }
}

// Both warpgroups take every key tile; warpgroup w its keys 64 w .. 64 w + 63.  Thread = query
// row of the tile; warp wq of warpgroup 0 and warp wq of warpgroup 1 hold the same 32 rows.
// Per item: the key tiles (the per-row values come from warps 2 and 3), and the output once the
// item's products have completed (then A, B, C and the item's sums are released).  Every named barrier is taken alike by all its warps, also after a failed wait (the
// work is then skipped); after a failure anywhere, the barrier at the end of the item's tiles
// tells every epilogue warp to stop.
__device__ void sm1_epilogue(const SmArgs& a, uint8_t* smem, Sm1Misc* ms, int w) {
  using CF = Sm1Cfg;
  const int wq = (threadIdx.x >> 5) & 3;
  const int r = wq * 32 + (threadIdx.x & 31);
  const uint32_t tl = ms->tmem + ((uint32_t)(wq * 32) << 16);
  constexpr float inv_sqrt_d = 0.125f;                      // d = 64
  constexpr float c2 = 1.4426950408889634f * inv_sqrt_d;   // log2(e) / sqrt(d)
  const int nt = (a.N + kT - 1) / kT;
  float* xmax = reinterpret_cast<float*>(smem + CF::XMAX_OFF);
  float2* stat = reinterpret_cast<float2*>(smem + CF::STAT_OFF);
  bool ok = true;
  int ex = 0;  // exchanges so far (alternating buffers), over all items
  int n0 = 0;  // the item's first key tile, counted over all items
  for (int it = 0; sm1_mine(it) < sm1_items(a); ++it) {
    const Sm1Item wi = sm1_item(a, sm1_mine(it));
    const int J = wi.J, par = it & 1;
    const int lim = a.causal ? wi.qt * kT + r : a.N - 1;  // last key of this query
    // last key visible to every row of this warp (uniform, as the aligned TMEM accesses require)
    const int lim_warp = a.causal ? wi.qt * kT + wq * 32 : a.N - 1;
    const int kn0 = wi.bh * nt;  // this sequence's first tile statistics record
    // the item's per-row values (gates, q_t . K_base, the bound factor of the logits: both warps
    // of a row pair read the one value, so that their exchange decisions below agree)
    if (ok) ok = mbar_wait_warp(&ms->cb_full[par], (it >> 1) & 1, &ms->abort);
    const float qn = reinterpret_cast<const float*>(smem + CF::ROWV_OFF)[(par * 5 + 4) * kT + r];
    if (!ok) ms->abort = 1;
    float m2 = -INFINITY, l = 0.0f;  // the row's reference (base-2 units), this half's exp-sum
    float2 xs = make_float2(0.0f, 0.0f);  // this half's sum of the last tile's bf16 logits
    // largest |k| of each tile (not needed for the first one: with the reference at -inf the
    // bound never holds there)
    float kn_next = 0.0f;
    // Every iteration takes the same exchange decisions in both warps of a row pair, also after
    // a failed wait (the work is then skipped), so that neither waits on the pair barrier in
    // vain.
    for (int g = 0; g < J; ++g) {
      const int n = n0 + g;
      const int b = n % CF::NB;
      const float kn = kn_next;
      if (g + 1 < J) kn_next = a.kstat[(size_t)(kn0 + g + 1) * kSmStat + 64];
      if (ok) {
        ok = mbar_wait_warp(&ms->s_full[b], (n / CF::NB) & 1, &ms->abort);
        if (!ok) ms->abort = 1;
      }
      const uint32_t ts = tl + sm1_sbuf(b) + 64 * w;  // this half's columns
      const int k0 = g * kT + 64 * w;                 // its first key
      const bool full = k0 + 63 <= lim_warp;
      const bool last = g == J - 1;
      uint32_t ra[32], rb[32];
      if (ok) {
        tc_fence_after();
        tmem_ld32_nowait(ts, ra);
        tmem_ld32_nowait(ts + 32, rb);
        tmem_wait_ld();
        reg_fence(ra);
        reg_fence(rb);
      }
      // ---- the reference rises only if some logit of the tile may exceed it by more than
      //      kRaise: c2 x <= c2 |q_t| max |k| (Cauchy-Schwarz) rules that out for most tiles;
      //      otherwise the two halves' maxima are exchanged (both warps decide alike) ----
      const bool exch = !__all_sync(0xffffffffu, qn * kn <= m2 + CF::kRaise);
      if (exch) {
        float cm = -INFINITY;
        if (!ok) {
        } else if (full) {
#pragma unroll
          for (int x = 0; x < 32; ++x)
            cm = fmaxf(cm, fmaxf(__uint_as_float(ra[x]), __uint_as_float(rb[x])));
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            if (k0 + x <= lim) cm = fmaxf(cm, __uint_as_float(ra[x]));
            if (k0 + 32 + x <= lim) cm = fmaxf(cm, __uint_as_float(rb[x]));
          }
        }
        float* xm = xmax + (ex & 1) * 2 * kT;
        ++ex;
        xm[w * kT + r] = cm;
        named_bar_sync(3 + wq, 64);
        const float tmx = fmaxf(xm[r], xm[kT + r]) * c2;
        const bool raise = tmx > m2 + CF::kRaise;  // false for a row without visible keys yet
        if (__any_sync(0xffffffffu, raise)) {
          const float f = (raise && m2 != -INFINITY) ? ex2(m2 - tmx) : 1.0f;
          if (raise) {
            l *= f;
            m2 = tmx;
          }
          if (ok && w == 0 && g >= 1) {
            // A's earlier tiles: wait until their products have completed (the commit that
            // frees tile n-1's stage follows them), then rescale
            ok = mbar_wait_warp(&ms->kv_empty[(n - 1) % CF::NS], ((n - 1) / CF::NS) & 1,
                                &ms->abort);
            if (!ok) ms->abort = 1;
            if (ok) {
              tc_fence_after();
#pragma unroll 1
              for (int q = 0; q < 4; ++q) {
                uint32_t av[16];
                tmem_ld16_nowait(tl + CF::TM_A + 16 * q, av);
                tmem_wait_ld();
                reg_fence(av);
#pragma unroll
                for (int y = 0; y < 16; ++y) av[y] = __float_as_uint(__uint_as_float(av[y]) * f);
                tmem_st16_nowait(tl + CF::TM_A + 16 * q, av);
              }
            }
          }
        }
      }
      if (!ok) continue;
      // ---- P = 2^{c2 x - m} and x as bf16 pairs over this half's own columns; the last tile's
      //      rounded logits are summed (the earlier tiles' sum comes from K_base) ----
      auto chunk_px = [&](const uint32_t (&rv)[32], const int ch) {
        float2 ls = make_float2(0.0f, 0.0f);
        if (full) {
          const float2 c2v = make_float2(c2, c2), nm = make_float2(-m2, -m2);
#pragma unroll
          for (int hp = 0; hp < 2; ++hp) {
            uint32_t pp[8], xp[8];
#pragma unroll
            for (int y = 0; y < 8; ++y) {
              const float2 xv = make_float2(__uint_as_float(rv[16 * hp + 2 * y]),
                                            __uint_as_float(rv[16 * hp + 2 * y + 1]));
              const float2 e = __ffma2_rn(xv, c2v, nm);
              const float2 pe = make_float2(ex2(e.x), ex2(e.y));
              ls = __fadd2_rn(ls, pe);
              pp[y] = pack_bf16x2(pe.x, pe.y);
              xp[y] = pack_bf16x2(xv.x, xv.y);
              if (last)
                xs = __fadd2_rn(xs, make_float2(__uint_as_float(xp[y] << 16),
                                                __uint_as_float(xp[y] & 0xffff0000u)));
            }
            tmem_st8_nowait(ts + 32 * ch + 16 * hp, pp);
            tmem_st8_nowait(ts + 32 * ch + 16 * hp + 8, xp);
          }
        } else {
#pragma unroll
          for (int hp = 0; hp < 2; ++hp) {
            uint32_t pp[8], xp[8];
#pragma unroll
            for (int y = 0; y < 8; ++y) {
              float pe[2], xe[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int x = 16 * hp + 2 * y + e;
                const float xv = __uint_as_float(rv[x]);
                const bool valid = k0 + 32 * ch + x <= lim;
                pe[e] = valid ? ex2(fmaf(xv, c2, -m2)) : 0.0f;
                xe[e] = valid ? xv : 0.0f;
              }
              ls.x += pe[0];
              ls.y += pe[1];
              pp[y] = pack_bf16x2(pe[0], pe[1]);
              xp[y] = pack_bf16x2(xe[0], xe[1]);
              if (last)
                xs = __fadd2_rn(xs, make_float2(__uint_as_float(xp[y] << 16),
                                                __uint_as_float(xp[y] & 0xffff0000u)));
            }
            tmem_st8_nowait(ts + 32 * ch + 16 * hp, pp);
            tmem_st8_nowait(ts + 32 * ch + 16 * hp + 8, xp);
          }
        }
        l += ls.x + ls.y;
      };
      chunk_px(ra, 0);
      chunk_px(rb, 1);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(&ms->w_full[b]);
    }
    // ---- the two halves' exp-sums (both relative to the row's common reference) and last-tile
    //      logit sums; every epilogue warp learns here whether any role has failed ----
    stat[w * kT + r] = make_float2(l, xs.x + xs.y);
    if (named_bar_any(1, 256, !ok || ms->abort != 0)) {
      ok = false;
      break;
    }
    const float2 s0 = stat[r], s1 = stat[kT + r];
    const float lt = s0.x + s1.x;
    // ---- the row's coefficients, while the last products complete; then the output:
    //      O = alpha A + beta B + gamma C, warpgroup w writing columns 32 w .. 32 w + 31 ----
    const Sm1Item wd = sm1_item(a, sm1_mine(it));
    const int t = wd.qt * kT + r;  // query index (0-based)
    const bool row_ok = t < a.N;
    const float tc = a.causal ? (float)(t + 1) : (float)a.N;
    const float* rowv = reinterpret_cast<const float*>(smem + CF::ROWV_OFF) + par * 5 * kT + r;
    float sig1 = 0.0f, sigh = 0.0f, sig0 = 0.0f;
    if (row_ok) {
      sig1 = sigmoid(rowv[0]);
      sigh = sigmoid(rowv[kT]);
      if (a.g0) sig0 = sigmoid(rowv[2 * kT]);
    }
    const float qk = rowv[3 * kT];
    const float rt = 1.0f / tc;
    const float alpha = lt > 0.0f ? sigh / lt : 0.0f;
    const float beta = (sig1 - sigh) * rt;
    const float Pt = (qk + s0.y + s1.y) * inv_sqrt_d;
    const float bs = beta * inv_sqrt_d;
    const float gamma = fmaf(-beta * Pt, rt, (sig0 - sigh) * rt);
    ok = mbar_wait_warp(&ms->o_full, par, &ms->abort);
    if (ok) {
      tc_fence_after();
      const int c0 = 32 * w;
      const float* cbase = reinterpret_cast<const float*>(smem + CF::CBASE_OFF) + par * 64 + c0;
      const uint32_t tcd = tl + sm1_sbuf((n0 + J - 1) % CF::NB);  // the diagonal tile's C
      float o[32];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {  // two 16-column rounds
        uint32_t av[16], bv[16], cv[16];
        tmem_ld16_nowait(tl + CF::TM_A + c0 + 16 * hh, av);
        tmem_ld16_nowait(tl + CF::TM_B + c0 + 16 * hh, bv);
        if (a.causal) tmem_ld16_nowait(tcd + c0 + 16 * hh, cv);
        tmem_wait_ld();
        reg_fence(av);
        reg_fence(bv);
        reg_fence(cv);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float c = cbase[16 * hh + j];
          if (a.causal) c += __uint_as_float(cv[j]);
          o[16 * hh + j] = fmaf(alpha, __uint_as_float(av[j]),
                                fmaf(bs, __uint_as_float(bv[j]), gamma * c));
        }
      }
      // the row's 64 output bytes as four 16-byte chunks, transposed within each group of four
      // lanes (rows 4g .. 4g + 3 of the warp) so that each store instruction writes whole 64-byte
      // row segments of eight rows rather than 16 bytes of 32 rows: afterwards lane 4g + j holds
      // chunk j of the row 4g + k in x[k]
      uint4 x[4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        x[q4] = make_uint4(pack_bf16x2(o[8 * q4 + 0], o[8 * q4 + 1]),
                           pack_bf16x2(o[8 * q4 + 2], o[8 * q4 + 3]),
                           pack_bf16x2(o[8 * q4 + 4], o[8 * q4 + 5]),
                           pack_bf16x2(o[8 * q4 + 6], o[8 * q4 + 7]));
      const int lane = (int)(threadIdx.x & 31), j = lane & 3;
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
      const int t4 = wd.qt * kT + wq * 32 + (lane & ~3);  // query index of the group's first row
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (t4 + k < a.N)
          *reinterpret_cast<uint4*>(out + ((size_t)wd.bh * a.N + t4 + k) * 64 + c0 + 8 * j) = x[k];
    } else {
      ms->abort = 1;
    }
    // A, B and C have been read (the next item's products and third S product may write them),
    // and so have the item's column sums
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
      mbar_arrive(&ms->acc_free);
      mbar_arrive(&ms->cb_empty[par]);
    }
    n0 += J;
  }
  if (!ok) report(a.status, kErrTimeout);
}

__global__ void __launch_bounds__(kSmThreads, 1) sm1_kernel(const __grid_constant__ SmParams p) {
  using CF = Sm1Cfg;
  const SmArgs& a = p.a;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (smem_u32(smem) & 1023u) {  // the swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) report(a.status, kErrUnsupported);
    return;
  }
  Sm1Misc* ms = reinterpret_cast<Sm1Misc*>(smem + CF::MISC_OFF);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&ms->q_full, 1);
    mbar_init(&ms->q_empty, 3);  // the item's last S product and warps 2, 3
    for (int i = 0; i < CF::NS; ++i) {
      mbar_init(&ms->kv_full[i], 1);
      mbar_init(&ms->kv_empty[i], 1);
    }
    for (int i = 0; i < CF::NB; ++i) {
      mbar_init(&ms->s_full[i], 1);
      mbar_init(&ms->w_full[i], 8);  // the 8 epilogue warps
    }
    mbar_init(&ms->o_full, 1);
    mbar_init(&ms->acc_free, 8);
    mbar_init(&ms->fin, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms->cb_full[i], 2);   // warps 2 and 3
      mbar_init(&ms->cb_empty[i], 8);  // the 8 epilogue warps
    }
    ms->abort = 0;
    ms->never = 0;
  }
  // the lower-triangular ones tile [query row][key] (K-major, two atoms of 64 keys: 1 where
  // key <= row), 128-byte swizzled
  for (int idx = threadIdx.x; idx < 2 * kT * 8; idx += kSmThreads) {
    const int part = idx / (kT * 8), rr = (idx / 8) % kT, c = idx % 8;
    uint32_t wv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int key0 = 64 * part + 8 * c + 2 * e;
      wv[e] = pack_bf16x2(key0 <= rr ? 1.0f : 0.0f, key0 + 1 <= rr ? 1.0f : 0.0f);
    }
    *reinterpret_cast<uint4*>(smem + CF::TRI_OFF + part * kAtom + sw128_off(rr, c)) =
        make_uint4(wv[0], wv[1], wv[2], wv[3]);
  }
  fence_proxy_async_smem();  // written by the threads, read by the tensor cores
  if (warp == 1) {
    tmem_alloc(&ms->tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 0) {
    if ((threadIdx.x & 31) == 0) sm1_producer(p, smem, ms);
  } else if (warp == 1) {
    sm1_mma(a, smem, ms);
  } else if (warp < 4) {
    sm1_colsum(a, smem, ms);
  } else {
    sm1_epilogue(a, smem, ms, (warp - 4) >> 2);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    // every MMA has completed once `fin` fires (it is committed after the last one)
    if (!mbar_wait(&ms->fin, 0, &ms->never, 4000000000ull)) report(a.status, kErrTimeout);
    tc_fence_after();
    tmem_dealloc(ms->tmem, 512);
  }
}

// Rotary map of the bf16 rows [BH, N, d] of q and of k (half-split pairs, token n at position
// n) into yq and yk, with the fp64-built (cos, sin) table [N][d/2]; the rotated values are
// rounded to bf16 once.  A thread takes 8 consecutive pairs of one row (16-byte loads and
// stores of each half); the first half of the threads does q, the second k.
__global__ void sm_rotate_kernel(const __nv_bfloat16* __restrict__ xq,
                                 const __nv_bfloat16* __restrict__ xk, __nv_bfloat16* __restrict__ yq,
                                 __nv_bfloat16* __restrict__ yk, const float2* __restrict__ table,
                                 int N, int d, size_t groups) {
  const int half = d / 2, gpr = half / 8;  // groups of 8 pairs per row
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < 2 * groups;
       i += (size_t)gridDim.x * blockDim.x) {
    const bool is_k = i >= groups;
    const size_t gi = is_k ? i - groups : i;
    const int a0 = (int)(gi % gpr) * 8;
    const size_t rowi = gi / gpr;  // (bh, n)
    const int n = (int)(rowi % N);
    const size_t o = rowi * d + a0;
    const __nv_bfloat16* x = is_k ? xk : xq;
    __nv_bfloat16* y = is_k ? yk : yq;
    const uint4 ua = *reinterpret_cast<const uint4*>(x + o);
    const uint4 ub = *reinterpret_cast<const uint4*>(x + o + half);
    const float4* tb = reinterpret_cast<const float4*>(table + (size_t)n * half + a0);
    const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
    uint32_t ra[4], rb[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {  // pairs a0 + 2e and a0 + 2e + 1
      const float4 cs = tb[e];     // (cos, sin) of both pairs
      float xa0, xa1, xb0, xb1;
      unpack_bf16x2(wa[e], xa0, xa1);
      unpack_bf16x2(wb[e], xb0, xb1);
      ra[e] = pack_bf16x2(__fmaf_rn(xa0, cs.x, -xb0 * cs.y), __fmaf_rn(xa1, cs.z, -xb1 * cs.w));
      rb[e] = pack_bf16x2(__fmaf_rn(xa0, cs.y, xb0 * cs.x), __fmaf_rn(xa1, cs.w, xb1 * cs.z));
    }
    *reinterpret_cast<uint4*>(y + o) = make_uint4(ra[0], ra[1], ra[2], ra[3]);
    *reinterpret_cast<uint4*>(y + o + half) = make_uint4(rb[0], rb[1], rb[2], rb[3]);
  }
}

// d = 64: CTAs of 512 threads walk the 128-token tiles of all (b, h): CTA c takes the tile
// position c % nt of the sequences c / nt, c / nt + S, ... (S CTAs per position, about two CTAs
// per SM in all), so that the rotary table entries of its rows are loaded once; each tile's q, k
// and v are brought in by TMA (128-byte swizzled, zero past the sequence) two tiles ahead, so
// that the loads of the next tiles run while this one is worked on.  Thread (row r = tid / 4, part p = tid % 4) takes the pairs 8 p .. 8 p + 7 of the tile's
// row r of k (and of q when rotating): columns 8 p .. 8 p + 7 and 32 + 8 p .. 32 + 8 p + 7.
// With a rotary table the row is rotated exactly as sm_rotate_kernel does it and rounded to bf16
// once; the statistics are those of the bf16 values the attention kernel reads: the 64 column
// sums of k and of v over the tile's keys (fp32; four 32-row partial sums, added in order), the
// largest row norm of k and the norm of every row of q.
struct PrepParams {
  CUtensorMap tq, tk, tv;  // q, k, v [B*H, N, 64] bf16, box {64, 128, 1}, 128-byte swizzle
  __nv_bfloat16* yq;
  __nv_bfloat16* yk;
  const float2* table;     // (cos, sin) [N][32], or null: no rotation
  float* kstat;
  int* status;
  int N, nt, BH, S;        // tiles per sequence, sequences, CTAs per tile position
};
struct PrepSmem {
  static constexpr uint32_t TILES = 0;                       // [2 buffers][q, k, v] atoms
  static constexpr uint32_t PART = 2 * 3 * kAtom;            // float [2][4][128] partial sums
  static constexpr uint32_t WMAX = PART + 2 * 4 * 128 * 4;   // float [2][16] warp maxima
  static constexpr uint32_t BAR = WMAX + 2 * 16 * 4;         // two mbarriers
  static constexpr uint32_t BYTES = BAR + 16;
};
constexpr int kPrepThreads = 512;

__global__ void __launch_bounds__(kPrepThreads) sm_prep_kernel(const __grid_constant__ PrepParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // the swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) report(p.status, kErrUnsupported);
    return;
  }
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + PrepSmem::BAR);
  const int tid = threadIdx.x, r = tid >> 2, pp = tid & 3;
  const bool rot = p.table != nullptr;
  const uint32_t base = smem_u32(smem) + PrepSmem::TILES;
  const int tile = (int)blockIdx.x % p.nt, bh0 = (int)blockIdx.x / p.nt;
  // thread 0: the q, k and v tiles of sequence bh into buffer b
  auto issue = [&](int bh, int b) {
    const uint32_t dst = base + (uint32_t)b * 3 * kAtom;
    mbar_arrive_expect_tx(&bar[b], 3 * kAtom);
    tma_load_3d(dst, &p.tq, 0, tile * kT, bh, &bar[b]);
    tma_load_3d(dst + kAtom, &p.tk, 0, tile * kT, bh, &bar[b]);
    tma_load_3d(dst + 2 * kAtom, &p.tv, 0, tile * kT, bh, &bar[b]);
  };
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
  }
  __syncthreads();
  if (tid == 0) {
    if (bh0 < p.BH) issue(bh0, 0);
    if (bh0 + p.S < p.BH) issue(bh0 + p.S, 1);
  }
  const int n = tile * kT + r;
  const bool valid = n < p.N;
  // (cos, sin) of this thread's pairs 8 p + 2 e, 8 p + 2 e + 1, the same for every sequence
  float4 cs[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    cs[e] = (rot && valid) ? reinterpret_cast<const float4*>(p.table + (size_t)n * 32 + 8 * pp)[e]
                           : make_float4(1.0f, 0.0f, 1.0f, 0.0f);
  int never = 0;
  for (int j = 0, bh = bh0; bh < p.BH; ++j, bh += p.S) {
    const int b = j & 1;
    const uint32_t qt = base + (uint32_t)b * 3 * kAtom, kt = qt + kAtom, vt = kt + kAtom;
    if (!mbar_wait(&bar[b], (j >> 1) & 1, &never)) report(p.status, kErrTimeout);
    uint4 ka = lds128(kt + sw128_off(r, pp)), kb = lds128(kt + sw128_off(r, 4 + pp));
    uint4 qa = lds128(qt + sw128_off(r, pp)), qb = lds128(qt + sw128_off(r, 4 + pp));
    if (rot && valid) {
      auto rotate = [&](uint4& ua, uint4& ub) {
        uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float xa0, xa1, xb0, xb1;
          unpack_bf16x2(wa[e], xa0, xa1);
          unpack_bf16x2(wb[e], xb0, xb1);
          wa[e] = pack_bf16x2(__fmaf_rn(xa0, cs[e].x, -xb0 * cs[e].y),
                              __fmaf_rn(xa1, cs[e].z, -xb1 * cs[e].w));
          wb[e] = pack_bf16x2(__fmaf_rn(xa0, cs[e].y, xb0 * cs[e].x),
                              __fmaf_rn(xa1, cs[e].w, xb1 * cs[e].z));
        }
        ua = make_uint4(wa[0], wa[1], wa[2], wa[3]);
        ub = make_uint4(wb[0], wb[1], wb[2], wb[3]);
      };
      rotate(ka, kb);
      rotate(qa, qb);
      const size_t off = ((size_t)bh * p.N + n) * 64 + 8 * pp;
      *reinterpret_cast<uint4*>(p.yq + off) = qa;
      *reinterpret_cast<uint4*>(p.yq + off + 32) = qb;
      *reinterpret_cast<uint4*>(p.yk + off) = ka;
      *reinterpret_cast<uint4*>(p.yk + off + 32) = kb;
      // the rotated row, for the column sums
      sts128(kt + sw128_off(r, pp), ka);
      sts128(kt + sw128_off(r, 4 + pp), kb);
    }
    // squared row norms of k and of q (this thread's 16 values, then the row); the norm of each
    // q row, and the tile's largest of k
    float n2 = 0.0f, q2 = 0.0f;
    {
      const uint32_t w8[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
      const uint32_t v8[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float x0, x1, y0, y1;
        unpack_bf16x2(w8[e], x0, x1);
        n2 = __fmaf_rn(x0, x0, n2);
        n2 = __fmaf_rn(x1, x1, n2);
        unpack_bf16x2(v8[e], y0, y1);
        q2 = __fmaf_rn(y0, y0, q2);
        q2 = __fmaf_rn(y1, y1, q2);
      }
    }
    n2 += __shfl_xor_sync(0xffffffffu, n2, 1);
    n2 += __shfl_xor_sync(0xffffffffu, n2, 2);
    q2 += __shfl_xor_sync(0xffffffffu, q2, 1);
    q2 += __shfl_xor_sync(0xffffffffu, q2, 2);
    if (pp == 0) p.kstat[((size_t)bh * p.nt + tile) * kSmStat + 132 + r] = sqrtf(q2);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) n2 = fmaxf(n2, __shfl_xor_sync(0xffffffffu, n2, o));
    float* wmax = reinterpret_cast<float*>(smem + PrepSmem::WMAX) + b * 16;
    float* part = reinterpret_cast<float*>(smem + PrepSmem::PART) + b * 4 * 128;
    if ((tid & 31) == 0) wmax[tid >> 5] = n2;
    __syncthreads();
    {
      const int c = tid & 127, qq = tid >> 7;  // column c of k (c < 64) or of v
      const uint32_t tt = c < 64 ? kt : vt;
      const int cc = c & 63;
      float sum = 0.0f;
#pragma unroll 8
      for (int rr = 32 * qq; rr < 32 * qq + 32; ++rr) {
        uint16_t h;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(tt + sw128_off(rr, cc >> 3) + 2 * (cc & 7)));
        sum += __uint_as_float((uint32_t)h << 16);
      }
      part[qq * 128 + c] = sum;
    }
    __syncthreads();  // every read of buffer b is done: it takes the tile after next
    if (tid == 0 && bh + 2 * p.S < p.BH) {
      fence_proxy_async_smem();
      issue(bh + 2 * p.S, b);
    }
    float* st = p.kstat + ((size_t)bh * p.nt + tile) * kSmStat;
    if (tid < 128) {
      st[tid < 64 ? tid : tid + 4] =
          ((part[tid] + part[128 + tid]) + part[256 + tid]) + part[384 + tid];
    } else if (tid == 128) {
      float m = wmax[0];
#pragma unroll
      for (int w = 1; w < 16; ++w) m = fmaxf(m, wmax[w]);
      st[64] = sqrtf(m);
    }
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn sm_encode_fn() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load();
  if (!f) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      f = reinterpret_cast<EncodeTiledFn>(ptr);
      fn.store(f);
    }
  }
  return f;
}

// [B*H, N, d] bf16 viewed as 3-D (d fastest), boxes {64, 128, 1}, 128-byte swizzle; rows past N
// read as zeros.
bool sm_map(CUtensorMap* m, const void* ptr, int d, int N, int BH) {
  EncodeTiledFn f = sm_encode_fn();
  if (!f) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * (cuuint64_t)d * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)kT, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_sm_d(const SmArgs& a, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_set{0};  // bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(sm_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SmCfg<D>::BYTES);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  SmParams p;
  p.a = a;
  const int BH = a.B * a.H;
  if (!sm_map(&p.tq, a.q, D, a.N, BH) || !sm_map(&p.tk, a.k, D, a.N, BH) ||
      !sm_map(&p.tv, a.v, D, a.N, BH))
    return cudaErrorNotSupported;
  const dim3 grid(BH, (a.N + kT - 1) / kT, 1);
  sm_kernel<D><<<grid, kSmThreads, SmCfg<D>::BYTES, stream>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_sm1(const SmArgs& a, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_set{0};  // bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(sm1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Sm1Cfg::BYTES);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  SmParams p;
  p.a = a;
  const int BH = a.B * a.H;
  if (!sm_map(&p.tq, a.q, 64, a.N, BH) || !sm_map(&p.tk, a.k, 64, a.N, BH) ||
      !sm_map(&p.tv, a.v, 64, a.N, BH))
    return cudaErrorNotSupported;
  // persistent: one CTA per SM (at most one per item)
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long items = (long long)BH * ((a.N + kT - 1) / kT);
  if (items > 0x7fffffffll) return cudaErrorInvalidValue;
  const int grid = (int)(items < sms ? items : sms);
  if (grid == 0) return cudaSuccess;
  sm1_kernel<<<grid, kSmThreads, Sm1Cfg::BYTES, stream>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

bool sm_supported(int d, int dtype) { return dtype == 0 && (d == 64 || d == 128); }

cudaError_t launch_sm_rotate(const void* q, const void* k, void* yq, void* yk,
                             const float2* table, int BH, int N, int d, cudaStream_t stream) {
  const size_t groups = (size_t)BH * N * (d / 16);  // 8 pairs per group, per tensor
  if (groups == 0) return cudaSuccess;
  const size_t want = (2 * groups + 255) / 256;
  const int blocks = (int)(want < 152 * 16 ? want : 152 * 16);
  sm_rotate_kernel<<<blocks, 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<__nv_bfloat16*>(yq), static_cast<__nv_bfloat16*>(yk), table, N, d, groups);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_sm_prep(const void* q, const void* k, const void* v, void* yq, void* yk,
                           const float2* table, float* kstat, int* status, int BH, int N,
                           cudaStream_t stream) {
  const int nt = (N + kT - 1) / kT;
  const long long ntiles = (long long)BH * nt;
  if (ntiles == 0) return cudaSuccess;
  if (ntiles > 0x7fffffffll) return cudaErrorInvalidValue;
  static std::atomic<uint64_t> attr_set{0};  // bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(sm_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)PrepSmem::BYTES);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  PrepParams p;
  if (!sm_map(&p.tq, q, 64, N, BH) || !sm_map(&p.tk, k, 64, N, BH) || !sm_map(&p.tv, v, 64, N, BH))
    return cudaErrorNotSupported;
  p.yq = static_cast<__nv_bfloat16*>(yq);
  p.yk = static_cast<__nv_bfloat16*>(yk);
  p.table = table;
  p.kstat = kstat;
  p.status = status;
  p.N = N;
  p.nt = nt;
  p.BH = BH;
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // S CTAs per tile position, about two CTAs per SM in all (at least one per position)
  const int S = std::max(1, std::min(BH, 2 * sms / nt));
  p.S = S;
  const long long grid = (long long)nt * S;
  if (grid > 0x7fffffffll) return cudaErrorInvalidValue;
  sm_prep_kernel<<<(unsigned)grid, kPrepThreads, PrepSmem::BYTES, stream>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_sm(const SmArgs& a, cudaStream_t stream) {
  if (a.d == 64) return launch_sm1(a, stream);
  if (a.d == 128) return launch_sm_d<128>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace zs
