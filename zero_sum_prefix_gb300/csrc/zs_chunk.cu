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
//   The scalars s, m, Et = E e^{-m}, P follow the canonical fp32 token order of zs_common.cuh
//   (bit-identical to the decode step).
//
// Warp roles (352 threads, one CTA per (b, h, value slice), one CTA per SM):
//   warp 10    (T) : TMA producer: q and k chunks land 128B-swizzled directly in the operand
//                    tiles, the value slice in a 64B-swizzled staging tile (two stages at d=64).
//   warps 0-3  (P) : per token row: rotate q/k in place (RoPE), norms, gates, row coefficients,
//                    column scalars and the scaled value tile Vsc.
//   warps 4-7  (E) : TMEM -> registers: masked Q K^T -> bf16 tile; state -> bf16 tile (and the
//                    F~ rescale); X -> output rows.
//   warp 8     (S) : the sequential scalar chain (prior-mean sums, logits, m, Et, P), 32 tokens
//                    per batch, running ahead of the other roles through a 2-slot ring.
//   warp 9     (M) : TMEM allocation; one elected thread issues every tcgen05.mma.
// TMEM (512 columns): [0,128) Q K^T, [128,256) X, [256, 256 + d) state^T.
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
constexpr int kThreads = 352;
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
  static constexpr uint32_t SCAL_OFF = COLS_OFF + NS * 3 * kC * 4;  // float [2][4][128]
  static constexpr uint32_t MISC_OFF = SCAL_OFF + 2 * 4 * kC * 4;
  static constexpr uint32_t BYTES = MISC_OFF + 512;
  static constexpr uint32_t SMEM = BYTES + 1024;                 // + alignment slack
  static constexpr uint32_t TM_A = 0, TM_X = 128, TM_ST = 256;
};

struct Misc {
  uint64_t tma_full[2];
  uint64_t scal_full[2], scal_empty[2];
  uint64_t op_full[2], op_empty[2];
  uint64_t a_full, a_free, am_full, sst_full, x_full, x_free, st_done, fin;
  float Mslot[2];
  float Mop[2];
  uint32_t tmem;
  int abort;
  int never;  // stays 0: lets the final TMEM-release wait ignore the abort flag
};

struct ChunkParams {
  CUtensorMap tq, tk, tv;  // q, k: box {64, 128, 1} 128B swizzle; v: box {32, 128, 1} 64B swizzle
  FwdArgs a;
};

__device__ __forceinline__ void fail_wait(Misc* ms, int* status) {
  report(status, kErrTimeout);
  ms->abort = 1;
}

// ============================================================================ S: scalar chain
template <int D>
__device__ void role_scalar(const FwdArgs& a, uint8_t* smem, Misc* ms, int bh, int h,
                            size_t row0, int nch) {
  constexpr int R = D / 32;
  const int lane = threadIdx.x & 31;
  const __nv_bfloat16* __restrict__ u = static_cast<const __nv_bfloat16*>(a.u) + row0 * D;
  float* ring = reinterpret_cast<float*>(smem + Cfg<D>::SCAL_OFF);
  const int N = a.N;
  const bool dbg = blockIdx.y == 0;
  const float etau = expf(a.tau[h]);
  const float sqrtd = __fsqrt_rn((float)D);
  float S[R], mu[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    S[r] = 0.0f;
    mu[r] = a.mu[(size_t)h * D + lane + 32 * r];
  }
  float m_c = -INFINITY, E_c = 0.0f, P_c = 0.0f;

  for (int c = 0; c < nch; ++c) {
    const int slot = c & 1;
    if (c >= 2 && !mbar_wait_warp(&ms->scal_empty[slot], ((c >> 1) - 1) & 1, &ms->abort)) {
      fail_wait(ms, a.status);
      return;
    }
    float* rs = ring + slot * 4 * kC;
    for (int b = 0; b < kC / 32; ++b) {
      const int i0 = c * kC + b * 32;
      // column chains: lane owns columns lane + 32 r; partial dot of every token of the batch
      float pp[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int i = i0 + j;
        // unconditional (clamped) loads so the whole batch can be in flight at once
        const int ic = i < N ? i : N - 1;
        float uu[R];
#pragma unroll
        for (int r = 0; r < R; ++r) uu[r] = __bfloat162float(u[(size_t)ic * D + lane + 32 * r]);
        if (i < N) {
#pragma unroll
          for (int r = 0; r < R; ++r) S[r] = __fadd_rn(S[r], uu[r]);
        } else {
#pragma unroll
          for (int r = 0; r < R; ++r) uu[r] = 0.0f;
        }
        float p = __fmul_rn(uu[0], __fmaf_rn(etau, mu[0], S[0]));
#pragma unroll
        for (int r = 1; r < R; ++r) p = __fmaf_rn(uu[r], __fmaf_rn(etau, mu[r], S[r]), p);
        pp[j] = p;
      }
      // transpose-reduce: the butterfly tree of zs_common.cuh for 32 tokens at once;
      // afterwards lane l holds the full dot of token i0 + l.
#pragma unroll
      for (int w = 16; w >= 1; w >>= 1) {
        const bool up = (lane & w) != 0;
#pragma unroll
        for (int k = 0; k < w; ++k) {
          const float send = up ? pp[k] : pp[k + w];
          const float keep = up ? pp[k + w] : pp[k];
          const float recv = __shfl_xor_sync(0xffffffffu, send, w);
          pp[k] = __fadd_rn(keep, recv);
        }
      }
      const int i = i0 + lane;
      const bool valid = i < N;
      const float den = __fmul_rn(__fadd_rn(etau, (float)(i + 1)), sqrtd);
      const float s = -__fdiv_rn(pp[0], den);
      if (valid && !isfinite(s)) report(a.status, kErrRange);
      // running maximum (exact under any order), then f = e^{m_prev - m}, g = e^{s - m}
      float mm = valid ? s : -INFINITY;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float x = __shfl_up_sync(0xffffffffu, mm, o);
        if (lane >= o) mm = fmaxf(mm, x);
      }
      mm = fmaxf(mm, m_c);
      float mprev = __shfl_up_sync(0xffffffffu, mm, 1);
      if (lane == 0) mprev = m_c;
      const float f = expf(__fsub_rn(mprev, mm));
      const float g = expf(__fsub_rn(s, mm));
      // the two sequential chains, in token order, evaluated redundantly by every lane
      float myE = 0.0f, myP = 0.0f;
      const int nvalid = min(32, N - i0);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float sj = __shfl_sync(0xffffffffu, s, j);
        const float fj = __shfl_sync(0xffffffffu, f, j);
        const float gj = __shfl_sync(0xffffffffu, g, j);
        if (j < nvalid) {
          P_c = __fadd_rn(P_c, sj);
          E_c = __fmaf_rn(E_c, fj, gj);
        }
        if (lane == j) {
          myE = E_c;
          myP = P_c;
        }
      }
      m_c = __shfl_sync(0xffffffffu, mm, 31);
      const int r = b * 32 + lane;
      rs[0 * kC + r] = s;
      rs[1 * kC + r] = mm;
      rs[2 * kC + r] = myE;
      rs[3 * kC + r] = myP;
      if (dbg && valid) {
        if (a.dbg_s) a.dbg_s[row0 + i] = s;
        if (a.dbg_E) a.dbg_E[row0 + i] = myE;
        if (a.dbg_P) a.dbg_P[row0 + i] = myP;
        if (a.dbg_m) a.dbg_m[row0 + i] = mm;
      }
    }
    if (lane == 0) ms->Mslot[slot] = m_c;
    mbar_arrive(&ms->scal_full[slot]);  // 32 arrivals: every lane releases its own writes
  }

  if (a.final_state && blockIdx.y == 0) {
    float* rec = record_ptr(a.final_state, bh, D);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      rec[rec_S(D) + lane + 32 * r] = S[r];
      rec[rec_mu(D) + lane + 32 * r] = mu[r];
    }
    if (lane == 0) {
      RecordHead* hd = reinterpret_cast<RecordHead*>(rec);
      hd->t = N;
      hd->m = m_c;
      hd->Et = E_c;
      hd->P = P_c;
      hd->etau = etau;
    }
  }
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

// ============================================================================ P: operands
// Rotates (RoPE) row r of a 128B-swizzled bf16 tile in place and returns its squared norm.
// Pairs are (a, a + D/2); cs holds (cos, sin) of the D/2 pairs of this row's position.
template <int D>
__device__ __forceinline__ float rotate_inplace(uint8_t* tile, int r, bool rope,
                                                const float4 (&cs)[D / 4]) {
  constexpr int HALF = D / 2;
  float ss = 0.0f;
#pragma unroll
  for (int g = 0; g < HALF / 8; ++g) {
    const int ca = 8 * g, cb = 8 * g + HALF;
    uint4* pa = reinterpret_cast<uint4*>(tile + (ca / 64) * kTile + sw128_off(r, (ca % 64) / 8));
    uint4* pb = reinterpret_cast<uint4*>(tile + (cb / 64) * kTile + sw128_off(r, (cb % 64) / 8));
    const uint4 lo = *pa, hi = *pb;
    float xa[8], xb[8];
    const uint32_t wl[4] = {lo.x, lo.y, lo.z, lo.w}, wh[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      unpack_bf16x2(wl[k], xa[2 * k], xa[2 * k + 1]);
      unpack_bf16x2(wh[k], xb[2 * k], xb[2 * k + 1]);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      ss = __fmaf_rn(xa[k], xa[k], ss);
      ss = __fmaf_rn(xb[k], xb[k], ss);
    }
    if (rope) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 t = cs[4 * g + k];  // (cos, sin) of pairs 8g+2k and 8g+2k+1
        const float a0 = xa[2 * k], b0 = xb[2 * k], a1 = xa[2 * k + 1], b1 = xb[2 * k + 1];
        xa[2 * k] = __fsub_rn(__fmul_rn(a0, t.x), __fmul_rn(b0, t.y));
        xb[2 * k] = __fadd_rn(__fmul_rn(a0, t.y), __fmul_rn(b0, t.x));
        xa[2 * k + 1] = __fsub_rn(__fmul_rn(a1, t.z), __fmul_rn(b1, t.w));
        xb[2 * k + 1] = __fadd_rn(__fmul_rn(a1, t.w), __fmul_rn(b1, t.z));
      }
      uint4 oa, ob;
      oa.x = pack_bf16x2(xa[0], xa[1]);
      oa.y = pack_bf16x2(xa[2], xa[3]);
      oa.z = pack_bf16x2(xa[4], xa[5]);
      oa.w = pack_bf16x2(xa[6], xa[7]);
      ob.x = pack_bf16x2(xb[0], xb[1]);
      ob.y = pack_bf16x2(xb[2], xb[3]);
      ob.z = pack_bf16x2(xb[4], xb[5]);
      ob.w = pack_bf16x2(xb[6], xb[7]);
      *pa = oa;
      *pb = ob;
    }
  }
  return ss;
}

template <int D>
__device__ void role_operands(const FwdArgs& a, uint8_t* smem, Misc* ms, size_t row0, int nch) {
  using CF = Cfg<D>;
  const int r = threadIdx.x;  // token row inside the chunk, 0..127
  const int N = a.N;
  const float* ring = reinterpret_cast<const float*>(smem + CF::SCAL_OFF);
  float4* coef = reinterpret_cast<float4*>(smem + CF::COEF_OFF);
  float* colsc = reinterpret_cast<float*>(smem + CF::COLS_OFF);

  for (int c = 0; c < nch; ++c) {
    const int st = c % CF::NS;
    const int i = c * kC + r;
    const bool valid = i < N;
    // loads that do not depend on the TMA tiles go out first
    float4 cs[D / 4];
    if (a.rope) {
      const float4* tab = reinterpret_cast<const float4*>(a.rope_table + (size_t)min(i, N - 1) * (D / 2));
#pragma unroll
      for (int x = 0; x < D / 4; ++x) cs[x] = __ldg(tab + x);
    }
    float g1 = 0.0f, gh = 0.0f;
    if (valid) {
      g1 = __ldg(a.g1 + row0 + i);
      gh = __ldg(a.gh + row0 + i);
    }
    if (!mbar_wait(&ms->tma_full[st], (c / CF::NS) & 1, &ms->abort)) {
      fail_wait(ms, a.status);
      return;
    }
    uint8_t* qt = smem + CF::Q_OFF + st * CF::KA * kTile;
    uint8_t* kt = smem + CF::K_OFF + st * CF::KA * kTile;
    const bool rot = a.rope != 0 && valid;
    const float qq = rotate_inplace<D>(qt, r, rot, cs);
    const float kk = rotate_inplace<D>(kt, r, rot, cs);
    // value slice of this token from the staging tile
    float vv[kDV];
    {
      const uint8_t* vst = smem + CF::VST_OFF + st * 128 * 64;
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const uint4 w = *reinterpret_cast<const uint4*>(vst + sw64_off(r, x));
        unpack_bf16x2(w.x, vv[8 * x + 0], vv[8 * x + 1]);
        unpack_bf16x2(w.y, vv[8 * x + 2], vv[8 * x + 3]);
        unpack_bf16x2(w.z, vv[8 * x + 4], vv[8 * x + 5]);
        unpack_bf16x2(w.w, vv[8 * x + 6], vv[8 * x + 7]);
      }
    }
    // scalars of this chunk from the S ring
    const int slot = c & 1;
    if (!mbar_wait(&ms->scal_full[slot], (c >> 1) & 1, &ms->abort)) {
      fail_wait(ms, a.status);
      return;
    }
    const float* rs = ring + slot * 4 * kC;
    const float s = rs[0 * kC + r], m = rs[1 * kC + r], Et = rs[2 * kC + r], P = rs[3 * kC + r];
    const float M = ms->Mslot[slot];
    mbar_arrive(&ms->scal_empty[slot]);

    const float kap = __fdiv_rn(1.0f, fmaxf(__fsqrt_rn(kk), 1e-12f));
    const float rho = __fdiv_rn(1.0f, fmaxf(__fsqrt_rn(qq), 1e-12f));
    float ce = 0.0f, cs1 = 0.0f, ck = 0.0f;
    float4 cf = make_float4(0.f, 0.f, 0.f, 0.f);
    if (valid) {
      ce = __fmul_rn(expf(__fsub_rn(s, M)), kap);
      cs1 = __fmul_rn(s, kap);
      ck = kap;
      const float sig1 = sigmoid(g1), sigh = sigmoid(gh);
      const float rt = __fdiv_rn(1.0f, (float)(i + 1));
      const float b0 = __fmul_rn(__fsub_rn(sig1, sigh), rt);
      const float ahat = __fmul_rn(__fdiv_rn(sigh, Et), expf(__fsub_rn(M, m)));
      cf.x = __fmul_rn(rho, ahat);
      cf.y = __fmul_rn(rho, b0);
      cf.z = -__fmul_rn(rho, __fadd_rn(__fmul_rn(__fmul_rn(b0, P), rt), __fmul_rn(sigh, rt)));
      if (!isfinite(cf.x) || !isfinite(ce)) report(a.status, kErrRange);
    }
    coef[st * kC + r] = cf;
    colsc[(st * 3 + 0) * kC + r] = ce;
    colsc[(st * 3 + 1) * kC + r] = cs1;
    colsc[(st * 3 + 2) * kC + r] = ck;
    if (r == 0) ms->Mop[st] = M;
    // Vsc row: atom 0 = [v | e v], atom 1 = [s' v | k v]
    uint8_t* vt = smem + CF::V_OFF + st * 2 * kTile;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      uint4 pv, pe, ps, pk;
      pv.x = pack_bf16x2(vv[8 * x + 0], vv[8 * x + 1]);
      pv.y = pack_bf16x2(vv[8 * x + 2], vv[8 * x + 3]);
      pv.z = pack_bf16x2(vv[8 * x + 4], vv[8 * x + 5]);
      pv.w = pack_bf16x2(vv[8 * x + 6], vv[8 * x + 7]);
      pe.x = pack_bf16x2(__fmul_rn(ce, vv[8 * x + 0]), __fmul_rn(ce, vv[8 * x + 1]));
      pe.y = pack_bf16x2(__fmul_rn(ce, vv[8 * x + 2]), __fmul_rn(ce, vv[8 * x + 3]));
      pe.z = pack_bf16x2(__fmul_rn(ce, vv[8 * x + 4]), __fmul_rn(ce, vv[8 * x + 5]));
      pe.w = pack_bf16x2(__fmul_rn(ce, vv[8 * x + 6]), __fmul_rn(ce, vv[8 * x + 7]));
      ps.x = pack_bf16x2(__fmul_rn(cs1, vv[8 * x + 0]), __fmul_rn(cs1, vv[8 * x + 1]));
      ps.y = pack_bf16x2(__fmul_rn(cs1, vv[8 * x + 2]), __fmul_rn(cs1, vv[8 * x + 3]));
      ps.z = pack_bf16x2(__fmul_rn(cs1, vv[8 * x + 4]), __fmul_rn(cs1, vv[8 * x + 5]));
      ps.w = pack_bf16x2(__fmul_rn(cs1, vv[8 * x + 6]), __fmul_rn(cs1, vv[8 * x + 7]));
      pk.x = pack_bf16x2(__fmul_rn(ck, vv[8 * x + 0]), __fmul_rn(ck, vv[8 * x + 1]));
      pk.y = pack_bf16x2(__fmul_rn(ck, vv[8 * x + 2]), __fmul_rn(ck, vv[8 * x + 3]));
      pk.z = pack_bf16x2(__fmul_rn(ck, vv[8 * x + 4]), __fmul_rn(ck, vv[8 * x + 5]));
      pk.w = pack_bf16x2(__fmul_rn(ck, vv[8 * x + 6]), __fmul_rn(ck, vv[8 * x + 7]));
      *reinterpret_cast<uint4*>(vt + sw128_off(r, x)) = pv;
      *reinterpret_cast<uint4*>(vt + sw128_off(r, 4 + x)) = pe;
      *reinterpret_cast<uint4*>(vt + kTile + sw128_off(r, x)) = ps;
      *reinterpret_cast<uint4*>(vt + kTile + sw128_off(r, 4 + x)) = pk;
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
    if (ok && c >= 1) ok = mbar_wait(&ms->x_free, (c - 1) & 1, &ms->abort);
    if (!ok) break;
    tc_fence_after();
    // ---- X[:, 0:96] = Q [F~ | G | H] (previous chunks); X[:, 96:128] = S V ----
    if (c >= 1) {
      const uint32_t sst = base + CF::SST_OFF + 32 * 128;  // state rows 32..127
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk / 4) * kTile + (kk % 4) * 32;
        mma_bf16(tX, sw128_desc(qt + off, 16, 1024), sw128_desc(sst + off, 16, 1024), id_qs,
                 kk > 0);
      }
    }
    const uint32_t sm = base + CF::AM_OFF;
#pragma unroll
    for (int kk = 0; kk < kC / 16; ++kk) {
      const uint32_t aoff = (kk / 4) * kTile + (kk % 4) * 32;  // K-major, K = token i
      const uint32_t boff = kk * 2048;                          // MN-major, 16 rows per step
      mma_bf16(tX + 96, sw128_desc(sm + aoff, 16, 1024), sw128_desc(vt + boff, kTile, 1024),
               id_sv, kk > 0);
    }
    mma_commit(&ms->x_full);
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

  for (int c = 0; c < nch && ok; ++c) {
    const int st = c % CF::NS;
    ok = mbar_wait_warp(&ms->op_full[st], (c / CF::NS) & 1, &ms->abort);
    if (!ok) break;
    const float4 cf = coef[st * kC + t];  // (a, b, g) of row t
    const float M_cur = ms->Mop[st];
    const float* ce = colsc + (st * 3 + 0) * kC;
    const float* cs = colsc + (st * 3 + 1) * kC;
    const float* ck = colsc + (st * 3 + 2) * kC;
    // ---- S = [i <= t] (Q K^T) (a e + b s' + g k), fp32 then bf16 (rows t, K = token i) ----
    ok = mbar_wait_warp(&ms->a_full, c & 1, &ms->abort);
    if (!ok) break;
    tc_fence_after();
    const uint32_t sm = base + CF::AM_OFF;
#pragma unroll
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
        const float ee[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
        const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
        const float kk[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
        float e[8];
#pragma unroll
        for (int y = 0; y < 8; ++y) {
          const float w = __fmaf_rn(cf.x, ee[y], __fmaf_rn(cf.y, ss[y], __fmul_rn(cf.z, kk[y])));
          const float val = __fmul_rn(v[x * 8 + y], w);
          e[y] = (cb < wq || col0 + y <= t) ? val : 0.0f;
        }
        uint4 p;
        p.x = pack_bf16x2(e[0], e[1]);
        p.y = pack_bf16x2(e[2], e[3]);
        p.z = pack_bf16x2(e[4], e[5]);
        p.w = pack_bf16x2(e[6], e[7]);
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
#pragma unroll
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
    // ---- X -> output row t ----
    ok = mbar_wait_warp(&ms->x_full, c & 1, &ms->abort);
    if (!ok) break;
    tc_fence_after();
    float xf[32], xg[32], xh[32], xs[32];
    tmem_ld32(tm + CF::TM_X + 96, xs);
    if (c >= 1) {
      tmem_ld32(tm + CF::TM_X + 0, xf);
      tmem_ld32(tm + CF::TM_X + 32, xg);
      tmem_ld32(tm + CF::TM_X + 64, xh);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) xf[j] = xg[j] = xh[j] = 0.0f;
    }
    tc_fence_before();
    mbar_arrive(&ms->x_free);
    const int i = c * kC + t;
    if (i < N) {
      uint4* dst = reinterpret_cast<uint4*>(out + (size_t)i * D + j0);
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        float o[8];
#pragma unroll
        for (int y = 0; y < 8; ++y) {
          const int j = 8 * x + y;
          o[y] = __fadd_rn(__fmaf_rn(cf.x, xf[j], __fmaf_rn(cf.y, xg[j], __fmul_rn(cf.z, xh[j]))),
                           xs[j]);
        }
        uint4 p;
        p.x = pack_bf16x2(o[0], o[1]);
        p.y = pack_bf16x2(o[2], o[3]);
        p.z = pack_bf16x2(o[4], o[5]);
        p.w = pack_bf16x2(o[6], o[7]);
        dst[x] = p;
      }
    }
    M_prev = M_cur;
  }
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
      mbar_init(&ms->scal_full[i], 32);
      mbar_init(&ms->scal_empty[i], 128);
      mbar_init(&ms->op_full[i], 128);
      mbar_init(&ms->op_empty[i], 1);
    }
    mbar_init(&ms->a_full, 1);
    mbar_init(&ms->a_free, 128);
    mbar_init(&ms->am_full, 128);
    mbar_init(&ms->sst_full, 128);
    mbar_init(&ms->x_full, 1);
    mbar_init(&ms->x_free, 128);
    mbar_init(&ms->st_done, 1);
    mbar_init(&ms->fin, 1);
    ms->abort = 0;
    ms->never = 0;
  }
  if (warp == 9) {
    tmem_alloc(&ms->tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp < 4) {
    role_operands<D>(a, smem, ms, row0, nch);
  } else if (warp < 8) {
    role_epilogue<D>(a, smem, ms, bh, row0, nch);
  } else if (warp == 8) {
    role_scalar<D>(a, smem, ms, bh, h, row0, nch);
  } else if (warp == 9) {
    if ((threadIdx.x & 31) == 0) role_mma<D>(a, smem, ms, nch);
  } else if ((threadIdx.x & 31) == 0) {
    role_tma<D>(p, smem, ms, bh, nch);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
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
      !make_map(&p.tv, a.v, D, a.N, BH, kDV, CU_TENSOR_MAP_SWIZZLE_64B))
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
