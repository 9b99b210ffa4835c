// Chunked tensor-core causal forward of the ZeroS layer (bf16 inputs, fp32 accumulation).
//
// Method: Paper-Notes "ZeroS: Zero-Sum Linear Attention for Efficient Transformers", method
// details: deviation logits, zero-sum weights w_{t,i} = sig1_t delta_{t,i}/t + sigh_t eps_{t,i},
// angular factor q_hat_t R_{t-i} k_hat_i^T, and the "linear-time prefix scan" with five states
// (E, P, F, G, H) giving o_t = q_hat_t (alpha_t F_t + beta_t G_t + gamma_t H_t).
//
// Chunked form used here (chunks of C = 128 tokens, value columns in slices of DV = 32):
//   w_{t,i} = alpha_t e^{s_i} + beta_t s_i + gamma_t, so with the chunk reference M_c (the
//   running maximum of s at the chunk's last token), Q = rot(q), K = rot(k) (bf16, unnormalised)
//   and rho_t = 1/|q_t|, kappa_i = 1/|k_i|, row coefficients (a, b, g)_t = rho_t (alphâ_t,
//   beta_t, gamma_t) with alphâ_t = sigh_t e^{M_c - m_t} / Et_t and column scalars
//   (e, s', k)_i = (e^{s_i - M_c} kappa_i, s_i kappa_i, kappa_i):
//     intra  S_{t,i} = [i <= t] (Q_t . K_i) (a_t e_i + b_t s'_i + g_t k_i)   (fp32, rounded once)
//     Vsc_i = [ v_i | e_i v_i | s'_i v_i | k_i v_i ]                          (C x 128, bf16)
//     X[:, 0:96]   = Q [F~ | G | H]   (state of the previous chunks)
//     X[:, 96:128] = S V
//     o_t = a_t X_F + b_t X_G + g_t X_H + X_SV
//     state^T (128 x d; rows [unused | F~ | G | H]) += Vsc^T K, F~ rescaled by
//     e^{M_{c-1} - M_c} before each chunk's update.
//   The weight is formed in fp32 before it is rounded: the three terms of w nearly cancel (the
//   weights sum to zero), so rounding them separately would amplify bf16 rounding errors.
//   The scalars s, m, Et = E e^{-m}, P follow the canonical blocked fp32 order of zs_common.cuh
//   (bit-identical to the decode step).
//
// Warp roles (448 threads, one CTA per (b, h, value slice), one CTA per SM):
//   warps 0-3   (PS): warp w owns the 32-token block w of the chunk: the block's column sums,
//                     logits and local scalar chains (carries of earlier blocks through shared
//                     memory, two bounded barriers per chunk); hands (s, m, Et, P) per token and
//                     the chunk reference to PO through a two-slot ring.
//   warps 4-7   (PO): per token row: rotary factors, rotate q/k in place (RoPE), norms, gates,
//                     row coefficients, column scalars and the scaled value tile Vsc.
//   warps 8-11  (E) : TMEM -> registers: S = masked (Q K^T) x weights -> bf16 tile; state ->
//                     bf16 tile (and the F~ rescale); X -> output rows.
//   warp 12     (M) : TMEM allocation; one elected thread issues every tcgen05.mma.
//   warp 13     (T) : TMA producers: lane 0 streams q and k chunks 128B-swizzled directly into
//                     the operand tiles and the value slice into a 64B-swizzled staging tile (two
//                     stages at d = 64); lane 1 streams each chunk's u rows (one buffer).
// TMEM (512 columns): [0,128) Q K^T, [128,384) X (two buffers, chunk parity), [384, 384 + d)
// state^T.
// Every mbarrier wait is bounded in time; a timeout records ZEROS_ERR_TIMEOUT, raises a CTA
// abort flag and every role leaves its loop; TMEM is released after the last MMA completes.
#include <math.h>

#include <atomic>

#include "zs_common.cuh"
#include "zs_internal.h"
#include "zs_sm100.cuh"

namespace zs {
namespace {

using namespace sm100;

constexpr int kC = 128;       // tokens per chunk
constexpr int kDV = 32;       // value columns per CTA
constexpr int kThreads = 448;
constexpr uint32_t kTile = 128 * 128;  // one [128 x 64] bf16 atom tile

template <int D>
struct Cfg {
  static constexpr int KA = D / 64;               // atom tiles along d
  static constexpr int NS = (D == 64) ? 2 : 1;    // operand stages
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t K_OFF = Q_OFF + NS * KA * kTile;
  static constexpr uint32_t V_OFF = K_OFF + NS * KA * kTile;
  static constexpr uint32_t VST_OFF = V_OFF + NS * 2 * kTile;    // raw v slices [NS][128 x 32]
  static constexpr uint32_t AM_OFF = VST_OFF + NS * 128 * 64;
  static constexpr uint32_t SST_OFF = AM_OFF + 2 * kTile;
  static constexpr uint32_t COEF_OFF = SST_OFF + KA * kTile;     // float4 [NS][128] row coefs
  static constexpr uint32_t COLS_OFF = COEF_OFF + NS * kC * 16;  // float [NS][3][128] columns
  static constexpr uint32_t U_OFF = COLS_OFF + NS * 3 * kC * 4;     // bf16 [128][D] u rows
  static constexpr uint32_t PHI_OFF = U_OFF + kC * D * 2;             // float [2][D/2] base angles
  static constexpr uint32_t THETA_OFF = PHI_OFF + 2 * (D / 2) * 4;    // float [D/2] frequencies
  static constexpr uint32_t LEND_OFF = THETA_OFF + (D / 2) * 4;       // float [4][D]
  static constexpr uint32_t BPUB_OFF = LEND_OFF + 4 * D * 4;         // float [4][4] + [2][4]
  static constexpr uint32_t CHAIN_OFF = BPUB_OFF + 128;               // float4 [4][32]
  static constexpr uint32_t SCAL_OFF = CHAIN_OFF + 4 * 32 * 16;     // float4 [2][128]
  static constexpr uint32_t MISC_OFF = SCAL_OFF + 2 * kC * 16;
  static constexpr uint32_t BYTES = MISC_OFF + 512;
  static constexpr uint32_t SMEM = BYTES + 1024;                 // + alignment slack
  static constexpr uint32_t TM_A = 0, TM_X = 128, TM_ST = 384;  // X: two buffers of 128
};

struct Misc {
  uint64_t tma_full[2];
  uint64_t u_full, u_empty;
  uint64_t op_full[2], op_empty[2];
  uint64_t a_full, a_free, am_full, sst_full, st_done, fin;
  uint64_t x_full[2], x_free[2];
  uint64_t pbar;   // reusable barrier of the four scalar warps (bounded waits)
  uint64_t pobar;  // reusable barrier of the four operand warps
  uint64_t scal_full[2], scal_empty[2];
  float Mop[2];
  float Mslot[2];
  uint32_t tmem;
  int abort;
  int never;  // stays 0: lets the final TMEM-release wait ignore the abort flag
};

struct ChunkParams {
  CUtensorMap tq, tk, tv;  // q, k: box {64, 128, 1} 128B swizzle; v: box {32, 128, 1} 64B swizzle
  CUtensorMap tu;          // u: box {d, 128, 1}, no swizzle (dense 2d-byte rows)
  FwdArgs a;
};

__device__ __forceinline__ void fail_wait(Misc* ms, int* status) {
  report(status, kErrTimeout);
  ms->abort = 1;
}

// ============================================================================ T: TMA producer
template <int D>
__device__ void role_tma(const ChunkParams& p, uint8_t* smem, Misc* ms, int bh, int nch) {
  using CF = Cfg<D>;
  const uint32_t base = smem_u32(smem);
  const int j0 = blockIdx.y * kDV;
  constexpr uint32_t bytes = 2 * CF::KA * kTile + 128 * 64;
  tma_prefetch_desc(&p.tq);
  tma_prefetch_desc(&p.tk);
  tma_prefetch_desc(&p.tv);
  for (int c = 0; c < nch; ++c) {
    const int st = c % CF::NS;
    if (c >= CF::NS && !mbar_wait(&ms->op_empty[st], ((c / CF::NS) - 1) & 1, &ms->abort)) {
      fail_wait(ms, p.a.status);
      return;
    }
    mbar_arrive_expect_tx(&ms->tma_full[st], bytes);
    const uint32_t qt = base + CF::Q_OFF + st * CF::KA * kTile;
    const uint32_t kt = base + CF::K_OFF + st * CF::KA * kTile;
#pragma unroll
    for (int at = 0; at < CF::KA; ++at) {
      tma_load_3d(qt + at * kTile, &p.tq, 64 * at, c * kC, bh, &ms->tma_full[st]);
      tma_load_3d(kt + at * kTile, &p.tk, 64 * at, c * kC, bh, &ms->tma_full[st]);
    }
    tma_load_3d(base + CF::VST_OFF + st * 128 * 64, &p.tv, j0, c * kC, bh, &ms->tma_full[st]);
  }
}

// u rows of each chunk (single buffer, released by the operand warps after their logits); a
// separate producer thread so that this stream never waits behind the operand stages.
template <int D>
__device__ void role_tma_u(const ChunkParams& p, uint8_t* smem, Misc* ms, int bh, int nch) {
  using CF = Cfg<D>;
  const uint32_t base = smem_u32(smem);
  tma_prefetch_desc(&p.tu);
  for (int c = 0; c < nch; ++c) {
    if (c >= 1 && !mbar_wait(&ms->u_empty, (c - 1) & 1, &ms->abort)) {
      fail_wait(ms, p.a.status);
      return;
    }
    mbar_arrive_expect_tx(&ms->u_full, kC * D * 2);
    tma_load_3d(base + CF::U_OFF, &p.tu, 0, c * kC, bh, &ms->u_full);
  }
}

// ============================================================================ P: operands
// Rotates (RoPE) pair group g (pairs 8g .. 8g+7 with partners + D/2) of row r of a
// 128B-swizzled bf16 tile in place and accumulates the row's squared norm into ss (two
// partial sums).  cs[k] = (cos, sin) of pair 8g + k.
template <int D>
__device__ __forceinline__ void rotate_group(uint8_t* tile, int r, int g, bool rope,
                                             const float2 (&cs)[8], float2& ss) {
  constexpr int HALF = D / 2;
  const int ca = 8 * g, cb = 8 * g + HALF;
  uint4* pa = reinterpret_cast<uint4*>(tile + (ca / 64) * kTile + sw128_off(r, (ca % 64) / 8));
  uint4* pb = reinterpret_cast<uint4*>(tile + (cb / 64) * kTile + sw128_off(r, (cb % 64) / 8));
  const uint4 lo = *pa, hi = *pb;
  const uint32_t wl[4] = {lo.x, lo.y, lo.z, lo.w}, wh[4] = {hi.x, hi.y, hi.z, hi.w};
  uint32_t oa[4], ob[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float2 xa, xb;  // elements (2k, 2k+1) of the two halves
    unpack_bf16x2(wl[k], xa.x, xa.y);
    unpack_bf16x2(wh[k], xb.x, xb.y);
    ss = __ffma2_rn(xa, xa, ss);
    ss = __ffma2_rn(xb, xb, ss);
    if (rope) {
      // pair (a, b) -> (a c - b s, a s + b c), one pair per component of the f32x2 ops
      const float2 c2 = make_float2(cs[2 * k].x, cs[2 * k + 1].x);
      const float2 s2 = make_float2(cs[2 * k].y, cs[2 * k + 1].y);
      const float2 na = __ffma2_rn(xa, c2, __fmul2_rn(make_float2(-xb.x, -xb.y), s2));
      const float2 nb = __ffma2_rn(xa, s2, __fmul2_rn(xb, c2));
      oa[k] = pack_bf16x2(na.x, na.y);
      ob[k] = pack_bf16x2(nb.x, nb.y);
    }
  }
  if (rope) {
    *pa = make_uint4(oa[0], oa[1], oa[2], oa[3]);
    *pb = make_uint4(ob[0], ob[1], ob[2], ob[3]);
  }
}

// The per-token scalars of one 32-token block, by the warp that owns the block (the canonical
// blocked order of zs_common.cuh).  Lane l owns columns R l + r while the column sums run; after
// the reduction lane j owns token j of the block.  Carries of the previous blocks arrive through
// shared memory (two bounded barriers among the four operand warps per chunk).
struct BlockCarry {
  float mC, EC, CP;
};

__device__ __forceinline__ void fold_block(BlockCarry& k, float LP, float ml, float El) {
  const float P = __fadd_rn(k.CP, LP);
  const float m = fmaxf(k.mC, ml);
  const float Et = __fmaf_rn(k.EC, expf(__fsub_rn(k.mC, m)), __fmul_rn(El, expf(__fsub_rn(ml, m))));
  k.CP = P;
  k.mC = m;
  k.EC = Et;
}

// Column values (R per lane) of token j of a 32-token block in the staged u tile.
template <int R>
struct UCols {
  float2 v[(R + 1) / 2];
};

template <int D>
__device__ __forceinline__ UCols<D / 32> load_ucols(const uint8_t* us, int j) {
  constexpr int R = D / 32;
  UCols<R> o;
  if (R == 1) {
    const uint16_t hv = *reinterpret_cast<const uint16_t*>(us + (size_t)j * D * 2);
    o.v[0] = make_float2(__uint_as_float((uint32_t)hv << 16), 0.0f);
  } else if (R == 2) {
    const uint32_t wv = *reinterpret_cast<const uint32_t*>(us + (size_t)j * D * 2);
    unpack_bf16x2(wv, o.v[0].x, o.v[0].y);
  } else {
    const uint2 wv = *reinterpret_cast<const uint2*>(us + (size_t)j * D * 2);
    unpack_bf16x2(wv.x, o.v[0].x, o.v[0].y);
    unpack_bf16x2(wv.y, o.v[(R + 1) / 2 - 1].x, o.v[(R + 1) / 2 - 1].y);
  }
  return o;
}

// ---------------------------------------------------------------- PS: scalars of the blocks
template <int D>
__device__ void role_scalars(const FwdArgs& a, uint8_t* smem, Misc* ms, int bh, int h,
                             size_t row0, int nch) {
  using CF = Cfg<D>;
  constexpr int R = D / 32;
  constexpr int RP = (R + 1) / 2;  // column pairs per lane (R = 1 uses the .x half only)
  const int r = threadIdx.x;       // token row inside the chunk, 0..127
  const int w = r >> 5, lane = r & 31;
  const int N = a.N;
  float* lend = reinterpret_cast<float*>(smem + CF::LEND_OFF);      // [4][D]
  float* bpub = reinterpret_cast<float*>(smem + CF::BPUB_OFF);      // [4][4] + kc [2][4]
  float4* chain = reinterpret_cast<float4*>(smem + CF::CHAIN_OFF);  // [4][32] (s, f, g, -)
  float4* scal = reinterpret_cast<float4*>(smem + CF::SCAL_OFF);    // [2][128] (s, m, Et, P)
  const bool dbg = blockIdx.y == 0;
  const float etau = expf(a.tau[h]);
  const float sqrtd = __fsqrt_rn((float)D);
  const float2 etau2 = make_float2(etau, etau);
  float2 mu2[RP], Cc[RP];
#pragma unroll
  for (int x = 0; x < RP; ++x) {
    mu2[x] = make_float2(a.mu[(size_t)h * D + R * lane + 2 * x],
                         R > 1 ? a.mu[(size_t)h * D + R * lane + 2 * x + 1] : 0.0f);
    Cc[x] = make_float2(0.0f, 0.0f);
  }
  if (r == 0) {
    bpub[16 + 0] = -INFINITY;  // chunk-start carries (mC, EC, CP) for chunk 0
    bpub[16 + 1] = 0.0f;
    bpub[16 + 2] = 0.0f;
  }

  for (int c = 0; c < nch; ++c) {
    const int slot = c & 1;
    const int i = c * kC + r;
    const bool valid = i < N;
    const int b0 = c * kC + 32 * w;  // first token of this warp's block
    const int nvalid = max(0, min(32, N - b0));
    // ---- u of the block from the staged tile: lane owns columns R lane .. R lane + R - 1 ----
    if (!mbar_wait_warp(&ms->u_full, c & 1, &ms->abort)) {
      fail_wait(ms, a.status);
      return;
    }
    const uint8_t* us = smem + CF::U_OFF + (size_t)(32 * w) * D * 2 + R * lane * 2;
    // ---- phase 1: local column sums of the block -> its end value ----
    float2 L[RP];
#pragma unroll
    for (int x = 0; x < RP; ++x) L[x] = make_float2(0.0f, 0.0f);
#pragma unroll 8
    for (int j = 0; j < 32; ++j) {
      const UCols<R> uj = load_ucols<D>(us, j);
#pragma unroll
      for (int x = 0; x < RP; ++x) L[x] = __fadd2_rn(L[x], uj.v[x]);
    }
#pragma unroll
    for (int x = 0; x < RP; ++x) {
      lend[w * D + R * lane + 2 * x] = L[x].x;
      if (R > 1) lend[w * D + R * lane + 2 * x + 1] = L[x].y;
    }
    mbar_arrive(&ms->pbar);
    if (!mbar_wait_warp(&ms->pbar, (2 * c) & 1, &ms->abort)) {
      fail_wait(ms, a.status);
      return;
    }
    // ---- column carry at this block's start (and at the next chunk's start) ----
    float2 Cw[RP];
#pragma unroll
    for (int ww = 0; ww < 4; ++ww) {
      if (ww == w) {
#pragma unroll
        for (int x = 0; x < RP; ++x) Cw[x] = Cc[x];
      }
#pragma unroll
      for (int x = 0; x < RP; ++x) {
        const float2 le = make_float2(lend[ww * D + R * lane + 2 * x],
                                      R > 1 ? lend[ww * D + R * lane + 2 * x + 1] : 0.0f);
        Cc[x] = __fadd2_rn(Cc[x], le);
      }
    }
    // ---- phase 2: S = C + L per token, logit partial products (two tokens per f32x2) ----
    float pp[32];
#pragma unroll
    for (int x = 0; x < RP; ++x) L[x] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const UCols<R> u0 = load_ucols<D>(us, j), u1 = load_ucols<D>(us, j + 1);
      float2 n0[RP], n1[RP];
#pragma unroll
      for (int x = 0; x < RP; ++x) {
        L[x] = __fadd2_rn(L[x], u0.v[x]);
        n0[x] = __ffma2_rn(etau2, mu2[x], __fadd2_rn(Cw[x], L[x]));
        L[x] = __fadd2_rn(L[x], u1.v[x]);
        n1[x] = __ffma2_rn(etau2, mu2[x], __fadd2_rn(Cw[x], L[x]));
      }
      // p = u[R l] n[R l], then fma over the lane's remaining columns, for tokens j and j + 1
      float2 p = __fmul2_rn(make_float2(u0.v[0].x, u1.v[0].x), make_float2(n0[0].x, n1[0].x));
#pragma unroll
      for (int col = 1; col < R; ++col) {
        const int x = col >> 1;
        const float a0 = (col & 1) ? u0.v[x].y : u0.v[x].x, a1 = (col & 1) ? u1.v[x].y : u1.v[x].x;
        const float m0 = (col & 1) ? n0[x].y : n0[x].x, m1 = (col & 1) ? n1[x].y : n1[x].x;
        p = __ffma2_rn(make_float2(a0, a1), make_float2(m0, m1), p);
      }
      pp[j] = p.x;
      pp[j + 1] = p.y;
    }
    mbar_arrive(&ms->u_empty);  // this thread is done with the staged u rows
    // transpose-reduce: the butterfly tree of the contract for 32 tokens at once; afterwards
    // lane j holds the full dot of token b0 + j.
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int k = 0; k < o; ++k) {
        const float send = up ? pp[k] : pp[k + o];
        const float keep = up ? pp[k + o] : pp[k];
        const float recv = __shfl_xor_sync(0xffffffffu, send, o);
        pp[k] = __fadd_rn(keep, recv);
      }
    }
    const float den = __fmul_rn(__fadd_rn(etau, (float)(i + 1)), sqrtd);
    const float s = -__fdiv_rn(pp[0], den);
    if (valid && !isfinite(s)) report(a.status, kErrRange);
    // ---- block-local running max, scaled exp-sum and logit sum (token order) ----
    float ml = valid ? s : -INFINITY;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float x = __shfl_up_sync(0xffffffffu, ml, o);
      if (lane >= o) ml = fmaxf(ml, x);
    }
    float mlp = __shfl_up_sync(0xffffffffu, ml, 1);
    if (lane == 0) mlp = -INFINITY;
    chain[w * 32 + lane] = make_float4(s, expf(__fsub_rn(mlp, ml)), expf(__fsub_rn(s, ml)), 0.0f);
    __syncwarp();
    float LP = 0.0f, El = 0.0f;
    const int kend = min(nvalid, lane + 1);  // this lane accumulates tokens 0 .. lane
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
      const float4 e = chain[w * 32 + k];
      if (k < kend) {
        LP = __fadd_rn(LP, e.x);
        El = __fmaf_rn(El, e.y, e.z);
      }
    }
    if (lane == 31) {  // block end values: tokens 0 .. nvalid-1
      bpub[w * 4 + 0] = LP;
      bpub[w * 4 + 1] = ml;
      bpub[w * 4 + 2] = El;
    }
    mbar_arrive(&ms->pbar);
    if (!mbar_wait_warp(&ms->pbar, (2 * c + 1) & 1, &ms->abort)) {
      fail_wait(ms, a.status);
      return;
    }
    // carries at this block's start: chunk-start carries folded over the earlier blocks
    const float* kcb = bpub + 16 + (c & 1) * 4;
    BlockCarry kw{kcb[0], kcb[1], kcb[2]};
    for (int ww = 0; ww < w; ++ww) fold_block(kw, bpub[ww * 4 + 0], bpub[ww * 4 + 1], bpub[ww * 4 + 2]);
    float M = kw.mC;  // running max at the chunk's last valid token (max is exact)
#pragma unroll
    for (int ww = 0; ww < 4; ++ww) M = fmaxf(M, bpub[ww * 4 + 1]);
    if (w == 3 && lane == 0) {  // chunk-start carries of the next chunk
      BlockCarry kn = kw;
      fold_block(kn, bpub[12 + 0], bpub[12 + 1], bpub[12 + 2]);
      float* kcn = bpub + 16 + ((c + 1) & 1) * 4;
      kcn[0] = kn.mC;
      kcn[1] = kn.EC;
      kcn[2] = kn.CP;
    }
    // this token's scalars
    const float P = __fadd_rn(kw.CP, LP);
    const float m = fmaxf(kw.mC, ml);
    const float Et = __fmaf_rn(kw.EC, expf(__fsub_rn(kw.mC, m)), __fmul_rn(El, expf(__fsub_rn(ml, m))));
    if (dbg && valid) {
      if (a.dbg_s) a.dbg_s[row0 + i] = s;
      if (a.dbg_E) a.dbg_E[row0 + i] = Et;
      if (a.dbg_P) a.dbg_P[row0 + i] = P;
      if (a.dbg_m) a.dbg_m[row0 + i] = m;
    }
    // hand the scalars to the operand warps (two-slot ring)
    if (c >= 2 && !mbar_wait_warp(&ms->scal_empty[slot], ((c >> 1) - 1) & 1, &ms->abort)) {
      fail_wait(ms, a.status);
      return;
    }
    scal[slot * kC + r] = make_float4(s, m, Et, P);
    if (r == 0) ms->Mslot[slot] = M;
    mbar_arrive(&ms->scal_full[slot]);
    // ---- recurrent state after the last token (prefill), by the warp owning that token ----
    if (a.final_state && dbg && c == nch - 1 && nvalid > 0 && b0 + nvalid == N) {
      float* rec = record_ptr(a.final_state, bh, D);
      const bool closed = nvalid == 32;  // the block is complete: fold it as the decode step does
      const float LPe = __shfl_sync(0xffffffffu, LP, 31);
      const float mle = __shfl_sync(0xffffffffu, ml, 31);
      const float Ele = __shfl_sync(0xffffffffu, El, 31);
      BlockCarry kf = kw;
      if (closed) fold_block(kf, LPe, mle, Ele);
#pragma unroll
      for (int x = 0; x < RP; ++x) {
#pragma unroll
        for (int y = 0; y < 2 && 2 * x + y < R; ++y) {
          const float cw = y ? Cw[x].y : Cw[x].x, le = y ? L[x].y : L[x].x;
          rec[rec_C(D) + R * lane + 2 * x + y] = closed ? __fadd_rn(cw, le) : cw;
          rec[rec_L(D) + R * lane + 2 * x + y] = closed ? 0.0f : le;
          rec[rec_mu(D) + R * lane + 2 * x + y] = y ? mu2[x].y : mu2[x].x;
        }
      }
      if (lane == 0) {
        RecordHead* hd = reinterpret_cast<RecordHead*>(rec);
        hd->t = N;
        hd->mC = kf.mC;
        hd->EC = kf.EC;
        hd->CP = kf.CP;
        hd->etau = etau;
        hd->ml = closed ? -INFINITY : mle;
        hd->El = closed ? 0.0f : Ele;
        hd->LP = closed ? 0.0f : LPe;
      }
    }
  }
}

// ---------------------------------------------------------------- PO: tensor-core operands
template <int D>
__device__ void role_operands(const FwdArgs& a, uint8_t* smem, Misc* ms, int h, size_t row0,
                              int nch) {
  using CF = Cfg<D>;
  const int r = threadIdx.x - 128;  // token row inside the chunk, 0..127
  const int w = r >> 5, lane = r & 31;
  const int N = a.N;
  float4* coef = reinterpret_cast<float4*>(smem + CF::COEF_OFF);
  float* colsc = reinterpret_cast<float*>(smem + CF::COLS_OFF);
  const float4* scal = reinterpret_cast<const float4*>(smem + CF::SCAL_OFF);
  float* phi = reinterpret_cast<float*>(smem + CF::PHI_OFF);      // [2][D/2]
  float* theta = reinterpret_cast<float*>(smem + CF::THETA_OFF);  // [D/2]
  const double two_pi = 6.283185307179586476925286766559;
  constexpr int PPW = (D / 2 + 3) / 4;  // rotary pairs per warp
  const int pj = w * PPW + lane;
  const bool owns_pair = a.rope && lane < PPW && pj < D / 2;
  double theta_d = 0.0;
  if (owns_pair) {
    theta_d = pow((double)a.rope_base, -2.0 * (double)pj / (double)D);
    theta[pj] = (float)theta_d;
  }

  for (int c = 0; c < nch; ++c) {
    const int st = c % CF::NS;
    const int slot = c & 1;
    const int i = c * kC + r;
    const bool valid = i < N;
    float g1 = 0.0f, gh = 0.0f;
    if (valid) {
      g1 = __ldg(a.g1 + row0 + i);
      gh = __ldg(a.gh + row0 + i);
    }
    // rotary base angle of this chunk per pair, reduced modulo 2 pi in fp64; token r of the
    // chunk then uses phi_j + r theta_j
    if (owns_pair) {
      const double ang = (double)(c * kC) * theta_d;
      phi[(c & 1) * (D / 2) + pj] = (float)(ang - rint(ang * (1.0 / two_pi)) * two_pi);
    }
    mbar_arrive(&ms->pobar);
    if (!mbar_wait_warp(&ms->pobar, c & 1, &ms->abort)) {
      fail_wait(ms, a.status);
      return;
    }
    // ---- rotate q, k in place (TMA tiles), norms ----
    if (!mbar_wait_warp(&ms->tma_full[st], (c / CF::NS) & 1, &ms->abort)) {
      fail_wait(ms, a.status);
      return;
    }
    uint8_t* qt = smem + CF::Q_OFF + st * CF::KA * kTile;
    uint8_t* kt = smem + CF::K_OFF + st * CF::KA * kTile;
    const bool rot = a.rope != 0 && valid;
    float2 qq2 = make_float2(0.0f, 0.0f), kk2 = make_float2(0.0f, 0.0f);
    const float* ph = phi + (c & 1) * (D / 2);
    const float rf = (float)r;
#pragma unroll 1
    for (int g = 0; g < D / 16; ++g) {
      float2 cs[8];
      if (rot) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          float sn, cn;
          __sincosf(__fmaf_rn(rf, theta[8 * g + k], ph[8 * g + k]), &sn, &cn);
          cs[k] = make_float2(cn, sn);
        }
      }
      rotate_group<D>(qt, r, g, rot, cs, qq2);
      rotate_group<D>(kt, r, g, rot, cs, kk2);
    }
    const float qq = __fadd_rn(qq2.x, qq2.y), kk = __fadd_rn(kk2.x, kk2.y);
    // value slice of this token from the staging tile
    float2 vv[kDV / 2];
    {
      const uint8_t* vst = smem + CF::VST_OFF + st * 128 * 64;
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const uint4 wv = *reinterpret_cast<const uint4*>(vst + sw64_off(r, x));
        unpack_bf16x2(wv.x, vv[4 * x + 0].x, vv[4 * x + 0].y);
        unpack_bf16x2(wv.y, vv[4 * x + 1].x, vv[4 * x + 1].y);
        unpack_bf16x2(wv.z, vv[4 * x + 2].x, vv[4 * x + 2].y);
        unpack_bf16x2(wv.w, vv[4 * x + 3].x, vv[4 * x + 3].y);
      }
    }
    // ---- scalars of this token from the scalar warps ----
    if (!mbar_wait_warp(&ms->scal_full[slot], (c >> 1) & 1, &ms->abort)) {
      fail_wait(ms, a.status);
      return;
    }
    const float4 sc = scal[slot * kC + r];
    const float M = ms->Mslot[slot];
    mbar_arrive(&ms->scal_empty[slot]);
    const float s = sc.x, m = sc.y, Et = sc.z, P = sc.w;
    // column scalars and row coefficients (these feed bf16 / fp32 products, not the scalar
    // contract: fast exp, reciprocal square root and division are accurate enough here)
    const float kap = rsqrtf(fmaxf(kk, 1e-24f));
    const float rho = rsqrtf(fmaxf(qq, 1e-24f));
    float ce = 0.0f, cs1 = 0.0f, ck = 0.0f;
    float4 cf = make_float4(0.f, 0.f, 0.f, 0.f);
    if (valid) {
      ce = __fmul_rn(__expf(__fsub_rn(s, M)), kap);
      cs1 = __fmul_rn(s, kap);
      ck = kap;
      const float sig1 = __fdividef(1.0f, 1.0f + __expf(-g1));
      const float sigh = __fdividef(1.0f, 1.0f + __expf(-gh));
      const float rt = __fdividef(1.0f, (float)(i + 1));
      const float b0c = (sig1 - sigh) * rt;
      const float ahat = __fdividef(sigh, Et) * __expf(M - m);
      cf.x = rho * ahat;
      cf.y = rho * b0c;
      cf.z = -rho * (b0c * P * rt + sigh * rt);
      if (!isfinite(cf.x) || !isfinite(ce)) report(a.status, kErrRange);
    }
    coef[st * kC + r] = cf;
    colsc[(st * 3 + 0) * kC + r] = ce;
    colsc[(st * 3 + 1) * kC + r] = cs1;
    colsc[(st * 3 + 2) * kC + r] = ck;
    if (r == 0) ms->Mop[st] = M;
    // Vsc row: atom 0 = [v | e v], atom 1 = [s' v | k v]
    uint8_t* vt = smem + CF::V_OFF + st * 2 * kTile;
    const float2 ce2 = make_float2(ce, ce), cs2 = make_float2(cs1, cs1), ck2 = make_float2(ck, ck);
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      uint32_t pv[4], pe[4], ps[4], pk[4];
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const float2 v2 = vv[4 * x + y];
        const float2 e2 = __fmul2_rn(ce2, v2), s2 = __fmul2_rn(cs2, v2), k2 = __fmul2_rn(ck2, v2);
        pv[y] = pack_bf16x2(v2.x, v2.y);
        pe[y] = pack_bf16x2(e2.x, e2.y);
        ps[y] = pack_bf16x2(s2.x, s2.y);
        pk[y] = pack_bf16x2(k2.x, k2.y);
      }
      *reinterpret_cast<uint4*>(vt + sw128_off(r, x)) = make_uint4(pv[0], pv[1], pv[2], pv[3]);
      *reinterpret_cast<uint4*>(vt + sw128_off(r, 4 + x)) = make_uint4(pe[0], pe[1], pe[2], pe[3]);
      *reinterpret_cast<uint4*>(vt + kTile + sw128_off(r, x)) = make_uint4(ps[0], ps[1], ps[2], ps[3]);
      *reinterpret_cast<uint4*>(vt + kTile + sw128_off(r, 4 + x)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    fence_proxy_async_smem();
    mbar_arrive(&ms->op_full[st]);
  }
}

// ============================================================================ M: MMA issue
template <int D>
__device__ void role_mma(const FwdArgs& a, uint8_t* smem, Misc* ms, int nch) {
  using CF = Cfg<D>;
  const uint32_t base = smem_u32(smem);
  const uint32_t tm = ms->tmem;
  const uint32_t tA = tm + CF::TM_A, tX = tm + CF::TM_X, tS = tm + CF::TM_ST;
  constexpr uint32_t id_qk = idesc_bf16_f32(128, 128, false, false);   // Q K^T
  constexpr uint32_t id_qs = idesc_bf16_f32(128, 96, false, false);    // Q [F|G|H]
  constexpr uint32_t id_sv = idesc_bf16_f32(128, 32, false, true);     // S V
  constexpr uint32_t id_st = idesc_bf16_f32(128, D, true, true);       // Vsc^T K
  bool ok = true;
  for (int c = 0; c < nch && ok; ++c) {
    const int st = c % CF::NS;
    const uint32_t qt = base + CF::Q_OFF + st * CF::KA * kTile;
    const uint32_t kt = base + CF::K_OFF + st * CF::KA * kTile;
    const uint32_t vt = base + CF::V_OFF + st * 2 * kTile;
    ok = mbar_wait(&ms->op_full[st], (c / CF::NS) & 1, &ms->abort);
    if (ok && c >= 1) ok = mbar_wait(&ms->a_free, (c - 1) & 1, &ms->abort);
    if (!ok) break;
    tc_fence_after();
    // ---- A = Q K^T (K = d) ----
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk / 4) * kTile + (kk % 4) * 32;
      mma_bf16(tA, sw128_desc(qt + off, 16, 1024), sw128_desc(kt + off, 16, 1024), id_qk,
               kk > 0);
    }
    mma_commit(&ms->a_full);
    ok = mbar_wait(&ms->am_full, c & 1, &ms->abort);
    if (ok && c >= 1) ok = mbar_wait(&ms->sst_full, (c - 1) & 1, &ms->abort);
    if (ok && c >= 2) ok = mbar_wait(&ms->x_free[c & 1], ((c >> 1) - 1) & 1, &ms->abort);
    if (!ok) break;
    tc_fence_after();
    const uint32_t tXc = tX + (uint32_t)(c & 1) * 128;
    // ---- X[:, 0:96] = Q [F~ | G | H] (previous chunks); X[:, 96:128] = S V ----
    if (c >= 1) {
      const uint32_t sst = base + CF::SST_OFF + 32 * 128;  // state rows 32..127
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk / 4) * kTile + (kk % 4) * 32;
        mma_bf16(tXc, sw128_desc(qt + off, 16, 1024), sw128_desc(sst + off, 16, 1024), id_qs,
                 kk > 0);
      }
    }
    const uint32_t sm = base + CF::AM_OFF;
#pragma unroll
    for (int kk = 0; kk < kC / 16; ++kk) {
      const uint32_t aoff = (kk / 4) * kTile + (kk % 4) * 32;  // K-major, K = token i
      const uint32_t boff = kk * 2048;                          // MN-major, 16 rows per step
      mma_bf16(tXc + 96, sw128_desc(sm + aoff, 16, 1024), sw128_desc(vt + boff, kTile, 1024),
               id_sv, kk > 0);
    }
    mma_commit(&ms->x_full[c & 1]);
    // ---- state^T += Vsc^T K (M = 128 value rows, N = d, K = chunk tokens) ----
#pragma unroll
    for (int kk = 0; kk < kC / 16; ++kk) {
      const uint32_t off = kk * 2048;
      mma_bf16(tS, sw128_desc(vt + off, kTile, 1024), sw128_desc(kt + off, kTile, 1024), id_st,
               (c > 0 || kk > 0) ? 1u : 0u);
    }
    mma_commit(&ms->st_done);
    mma_commit(&ms->op_empty[st]);
  }
  if (!ok) fail_wait(ms, a.status);
  mma_commit(&ms->fin);
}

// ============================================================================ E: epilogue
template <int D>
__device__ void role_epilogue(const FwdArgs& a, uint8_t* smem, Misc* ms, int bh, size_t row0,
                              int nch) {
  using CF = Cfg<D>;
  const int wq = (threadIdx.x >> 5) & 3;          // TMEM lane quadrant of this warp
  const int t = wq * 32 + (threadIdx.x & 31);     // TMEM lane = token row / state row
  const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
  const uint32_t tm = ms->tmem + lane_off;
  const uint32_t base = smem_u32(smem);
  const float4* coef = reinterpret_cast<const float4*>(smem + CF::COEF_OFF);
  const float* colsc = reinterpret_cast<const float*>(smem + CF::COLS_OFF);
  const int j0 = blockIdx.y * kDV;
  const int N = a.N;
  __nv_bfloat16* __restrict__ out = static_cast<__nv_bfloat16*>(a.out) + row0 * D;
  float M_prev = 0.0f;
  bool ok = true;
  float4 cf_prev = make_float4(0.f, 0.f, 0.f, 0.f);
  // o = X_SV + a X_F + b X_G + g X_H for chunk cc, one 32-column block at a time
  auto xstep = [&](int cc, const float4 cfc) -> bool {
    const int xb_par = cc & 1;
    if (!mbar_wait_warp(&ms->x_full[xb_par], (cc >> 1) & 1, &ms->abort)) return false;
    tc_fence_after();
    const uint32_t tx = tm + CF::TM_X + (uint32_t)xb_par * 128;
    float o[32];
    tmem_ld32(tx + 96, o);
    if (cc >= 1) {
      float xb[32];
      tmem_ld32(tx + 0, xb);
#pragma unroll
      for (int j = 0; j < 32; ++j) o[j] = __fmaf_rn(cfc.x, xb[j], o[j]);
      tmem_ld32(tx + 32, xb);
#pragma unroll
      for (int j = 0; j < 32; ++j) o[j] = __fmaf_rn(cfc.y, xb[j], o[j]);
      tmem_ld32(tx + 64, xb);
#pragma unroll
      for (int j = 0; j < 32; ++j) o[j] = __fmaf_rn(cfc.z, xb[j], o[j]);
    }
    tc_fence_before();
    mbar_arrive(&ms->x_free[xb_par]);
    const int i = cc * kC + t;
    if (i < N) {
      uint4* dst = reinterpret_cast<uint4*>(out + (size_t)i * D + j0);
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        uint4 p;
        p.x = pack_bf16x2(o[8 * x + 0], o[8 * x + 1]);
        p.y = pack_bf16x2(o[8 * x + 2], o[8 * x + 3]);
        p.z = pack_bf16x2(o[8 * x + 4], o[8 * x + 5]);
        p.w = pack_bf16x2(o[8 * x + 6], o[8 * x + 7]);
        dst[x] = p;
      }
    }
    return true;
  };

  for (int c = 0; c < nch && ok; ++c) {
    const int st = c % CF::NS;
    ok = mbar_wait_warp(&ms->op_full[st], (c / CF::NS) & 1, &ms->abort);
    if (!ok) break;
    const float4 cf = coef[st * kC + t];  // (a, b, g) of row t
    const float2 ra2 = make_float2(cf.x, cf.x), rb2 = make_float2(cf.y, cf.y),
                 rg2 = make_float2(cf.z, cf.z);
    const float M_cur = ms->Mop[st];
    const float* ce = colsc + (st * 3 + 0) * kC;
    const float* cs = colsc + (st * 3 + 1) * kC;
    const float* ck = colsc + (st * 3 + 2) * kC;
    // ---- S = [i <= t] (Q K^T) (a e + b s' + g k), fp32 then bf16 (rows t, K = token i) ----
    ok = mbar_wait_warp(&ms->a_full, c & 1, &ms->abort);
    if (!ok) break;
    tc_fence_after();
    const uint32_t sm = base + CF::AM_OFF;
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
      if (cb > wq) {  // every column of this block is after every row of this warp
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int col0 = cb * 32 + x * 8;
          sts128(sm + (col0 / 64) * kTile + sw128_off(t, (col0 % 64) / 8), make_uint4(0, 0, 0, 0));
        }
        continue;
      }
      float v[32];
      tmem_ld32(tm + CF::TM_A + cb * 32, v);
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int col0 = cb * 32 + x * 8;
        const float4 e0 = *reinterpret_cast<const float4*>(ce + col0);
        const float4 e1 = *reinterpret_cast<const float4*>(ce + col0 + 4);
        const float4 s0 = *reinterpret_cast<const float4*>(cs + col0);
        const float4 s1 = *reinterpret_cast<const float4*>(cs + col0 + 4);
        const float4 k0 = *reinterpret_cast<const float4*>(ck + col0);
        const float4 k1 = *reinterpret_cast<const float4*>(ck + col0 + 4);
        const float2 ee[4] = {make_float2(e0.x, e0.y), make_float2(e0.z, e0.w),
                              make_float2(e1.x, e1.y), make_float2(e1.z, e1.w)};
        const float2 ss[4] = {make_float2(s0.x, s0.y), make_float2(s0.z, s0.w),
                              make_float2(s1.x, s1.y), make_float2(s1.z, s1.w)};
        const float2 kk[4] = {make_float2(k0.x, k0.y), make_float2(k0.z, k0.w),
                              make_float2(k1.x, k1.y), make_float2(k1.z, k1.w)};
        uint32_t pw[4];
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const float2 wgt = __ffma2_rn(ra2, ee[y], __ffma2_rn(rb2, ss[y], __fmul2_rn(rg2, kk[y])));
          float2 val = __fmul2_rn(make_float2(v[x * 8 + 2 * y], v[x * 8 + 2 * y + 1]), wgt);
          if (cb == wq) {  // diagonal block: keep i <= t only
            if (col0 + 2 * y > t) val.x = 0.0f;
            if (col0 + 2 * y + 1 > t) val.y = 0.0f;
          }
          pw[y] = pack_bf16x2(val.x, val.y);
        }
        const uint4 p = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        sts128(sm + (col0 / 64) * kTile + sw128_off(t, (col0 % 64) / 8), p);
      }
    }
    tc_fence_before();
    mbar_arrive(&ms->a_free);
    fence_proxy_async_smem();
    mbar_arrive(&ms->am_full);
    // ---- state (after chunk c-1) -> bf16 B operand rows 32..127, F~ rescaled to M_c ----
    if (c >= 1) {
      ok = mbar_wait_warp(&ms->st_done, (c - 1) & 1, &ms->abort);
      if (!ok) break;
      tc_fence_after();
      if (wq >= 1) {
        const bool rescale = (wq == 1) && (M_cur > M_prev);
        const float fac = rescale ? expf(__fsub_rn(M_prev, M_cur)) : 1.0f;
        const uint32_t sst = base + CF::SST_OFF;
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
          float v[32];
          tmem_ld32(tm + CF::TM_ST + cb * 32, v);
          if (rescale) {
#pragma unroll
            for (int y = 0; y < 32; ++y) v[y] = __fmul_rn(v[y], fac);
            tmem_st32(tm + CF::TM_ST + cb * 32, v);
          }
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            uint4 p;
            p.x = pack_bf16x2(v[8 * x + 0], v[8 * x + 1]);
            p.y = pack_bf16x2(v[8 * x + 2], v[8 * x + 3]);
            p.z = pack_bf16x2(v[8 * x + 4], v[8 * x + 5]);
            p.w = pack_bf16x2(v[8 * x + 6], v[8 * x + 7]);
            const int col0 = cb * 32 + x * 8;
            sts128(sst + (col0 / 64) * kTile + sw128_off(t, (col0 % 64) / 8), p);
          }
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(&ms->sst_full);
    }
    // ---- output rows of the previous chunk (its X was computed while this chunk's S and
    // state tiles were being formed) ----
    if (c >= 1) {
      ok = xstep(c - 1, cf_prev);
      if (!ok) break;
    }
    cf_prev = cf;
    M_prev = M_cur;
  }
  if (ok && nch > 0) ok = xstep(nch - 1, cf_prev);
  if (!ok) {
    fail_wait(ms, a.status);
    return;
  }
  // ---- final state (prefill): columns j0.. of F~, G, H (state rows 32..127) ----
  if (a.final_state && nch > 0) {
    if (!mbar_wait_warp(&ms->st_done, (nch - 1) & 1, &ms->abort)) {
      fail_wait(ms, a.status);
      return;
    }
    tc_fence_after();
    if (wq >= 1) {
      float* rec = record_ptr(a.final_state, bh, D);
      const int j = t % 32;
      const int off = wq == 1 ? rec_F(D) : wq == 2 ? rec_G(D) : rec_H(D);
#pragma unroll
      for (int cb = 0; cb < D / 32; ++cb) {
        float v[32];
        tmem_ld32(tm + CF::TM_ST + cb * 32, v);
#pragma unroll
        for (int y = 0; y < 32; ++y) rec[off + (cb * 32 + y) * D + j0 + j] = v[y];
      }
    }
  }
}

// ============================================================================ kernel
template <int D>
__global__ void __launch_bounds__(kThreads, 1) chunk_kernel(const __grid_constant__ ChunkParams p) {
  using CF = Cfg<D>;
  const FwdArgs& a = p.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Misc* ms = reinterpret_cast<Misc*>(smem + CF::MISC_OFF);
  const int warp = threadIdx.x >> 5;
  const int bh = blockIdx.x, h = bh % a.H;
  const size_t row0 = (size_t)bh * a.N;
  const int nch = (a.N + kC - 1) / kC;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms->tma_full[i], 1);
      mbar_init(&ms->op_full[i], 128);
      mbar_init(&ms->op_empty[i], 1);
    }
    mbar_init(&ms->a_full, 1);
    mbar_init(&ms->a_free, 128);
    mbar_init(&ms->am_full, 128);
    mbar_init(&ms->sst_full, 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms->x_full[i], 1);
      mbar_init(&ms->x_free[i], 128);
    }
    mbar_init(&ms->st_done, 1);
    mbar_init(&ms->fin, 1);
    mbar_init(&ms->pbar, 128);
    mbar_init(&ms->pobar, 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms->scal_full[i], 128);
      mbar_init(&ms->scal_empty[i], 128);
    }
    mbar_init(&ms->u_full, 1);
    mbar_init(&ms->u_empty, 128);
    ms->abort = 0;
    ms->never = 0;
  }
  if (warp == 12) {
    tmem_alloc(&ms->tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp < 4) {
    role_scalars<D>(a, smem, ms, bh, h, row0, nch);
  } else if (warp < 8) {
    role_operands<D>(a, smem, ms, h, row0, nch);
  } else if (warp < 12) {
    role_epilogue<D>(a, smem, ms, bh, row0, nch);
  } else if (warp == 12) {
    if ((threadIdx.x & 31) == 0) role_mma<D>(a, smem, ms, nch);
  } else if ((threadIdx.x & 31) == 0) {
    role_tma<D>(p, smem, ms, bh, nch);
  } else if ((threadIdx.x & 31) == 1) {
    role_tma_u<D>(p, smem, ms, bh, nch);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    // every MMA has completed once `fin` fires (it is committed after the last one)
    if (!mbar_wait(&ms->fin, 0, &ms->never, 4000000000ull)) report(a.status, kErrTimeout);
    tc_fence_after();
    tmem_dealloc(ms->tmem, 512);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

// [B*H, N, d] bf16 tensor viewed as 3-D (d fastest); boxes of {box_x, 128 tokens, 1 sequence}.
// Rows past N are filled with zeros by the copy engine.
bool make_map(CUtensorMap* m, const void* ptr, int d, int N, int BH, int box_x,
              CUtensorMapSwizzle sw) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * (cuuint64_t)d * 2};
  const cuuint32_t box[3] = {(cuuint32_t)box_x, (cuuint32_t)kC, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_d(const FwdArgs& a, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_set{0};  // bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(chunk_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Cfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  ChunkParams p;
  p.a = a;
  const int BH = a.B * a.H;
  if (!make_map(&p.tq, a.q, D, a.N, BH, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&p.tk, a.k, D, a.N, BH, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&p.tv, a.v, D, a.N, BH, kDV, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map(&p.tu, a.u, D, a.N, BH, D, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorNotSupported;
  dim3 grid(BH, D / kDV);
  chunk_kernel<D><<<grid, kThreads, Cfg<D>::SMEM, stream>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

bool chunk_supported(int d, int dtype, int causal) {
  return dtype == 0 && causal == 1 && (d == 64 || d == 128);
}

cudaError_t launch_fwd_chunk(const FwdArgs& a, cudaStream_t stream) {
  if (a.d == 64) return launch_d<64>(a, stream);
  if (a.d == 128) return launch_d<128>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace zs
