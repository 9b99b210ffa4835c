// Chunked tensor-core causal forward of the ZeroS layer (bf16 inputs, fp16 operands, fp32
// accumulation).
//
// Method: Paper-Notes "ZeroS: Zero-Sum Linear Attention for Efficient Transformers", method
// details: deviation logits, zero-sum weights w_{t,i} = sig1_t delta_{t,i}/t + sigh_t eps_{t,i},
// angular factor q_hat_t R_{t-i} k_hat_i^T, and the "linear-time prefix scan" with five states
// (E, P, F, G, H) giving o_t = q_hat_t (alpha_t F_t + beta_t G_t + gamma_t H_t).
//
// Chunked form used here (chunks of C = 128 tokens, value columns in slices of DV = 32):
//   w_{t,i} = alpha_t e^{s_i} + beta_t s_i + gamma_t, so with the chunk reference M_c (the
//   running maximum of s at the chunk's last token), Q = rot(q), K = rot(k) (fp16,
//   unnormalised) and rho_t = 1/|q_t|, kappa_i = 1/|k_i|, row coefficients (a, b, g)_t =
//   rho_t (alphâ_t, beta_t, gamma_t) with alphâ_t = sigh_t e^{M_c - m_t} / Et_t and column
//   scalars (e, s', k)_i = (e^{s_i - M_c} kappa_i, s_i kappa_i, kappa_i):
//     W_{t,i} = a_t e_i + b_t s'_i + g_t k_i        (tensor core, hi/lo bf16 split, fp32 sum)
//     intra  S_{t,i} = [i <= t] (Q_t . K_i) W_{t,i} (fp32 product, times 2^kr_t, then fp16)
//     Vsc_i = [ v_i | e_i v_i | s'_i 2^-ks v_i | k_i v_i ]                    (C x 128, fp16)
//     X[:, 0:96]   = Q [F~ | G | H]   (state of the previous chunks, fp16 copy times 2^-kb)
//     X[:, 96:128] = S V
//     o_t = a'_t X_F + b'_t X_G + g'_t X_H + 2^-kr_t X_SV
//     state^T (128 x d; rows [unused | F~ | G | H]) += Vsc^T K, F~ rescaled by
//     e^{M_{c-1} - M_c} before each chunk's update.
//   The output coefficients a', b', g' carry the copy's 2^kb (and b' G's 2^ks); the copy keeps
//   F~ at the running maximum before the chunk, and a' takes e^{M_{c-1} - m_t} (power-of-two
//   range scales: zs_range.cuh).  q, k and v must lie within the fp16 range once rotated
//   (|x| < 45056 for q and k, |v| <= 65504), which is reported otherwise.
//   The weight is formed to fp32 accuracy before the product is rounded: the three terms of w
//   nearly cancel (the weights sum to zero), so rounding them separately would amplify the
//   operand rounding.  The scalars s, m, Et = E e^{-m}, P of every token come from the scalar
//   pass (zs_scalars.cu, the canonical blocked fp32 order of zs_common.cuh), which runs first;
//   the chunk reference M_c is the m of the chunk's last token.
//
// Warp roles (448 threads, one CTA per (b, h, value slice), one CTA per SM):
//   warps 0-7   (O) : operands; token row r = 32 (w % 4) + lane, half hf = w / 4 of the row's
//                     work: rotary factors and in-place rotation (RoPE) of the hf-th half of the
//                     rotary pairs of q and k (TMA-landed tiles), partial norms exchanged through
//                     shared memory; hf = 0 forms the row coefficients and the row weight
//                     operand, hf = 1 the column weight operand; each half builds half of the
//                     row's scaled value tile Vsc.
//   warps 8-11  (E) : TMEM -> registers: S = masked (Q K^T) o W -> fp16 tile; state -> fp16
//                     tile (and the F~ rescale); X -> output rows.
//   warp 12     (M) : TMEM allocation; the whole warp runs the issue loop (warp-uniform
//                     operands) and one elected lane issues every tcgen05.mma.
//   warp 13     (T) : TMA producer: q and k chunks 128B-swizzled directly into the operand
//                     tiles (two stages at d = 64) and the value slice into a 64B-swizzled
//                     staging tile, with an L2 prefetch of each chunk issued before its stage
//                     frees.
// TMEM (512 columns): [0,128) Q K^T, [128,256) W, [256,384) X, [384, 384 + d) state^T.
// Every mbarrier wait is bounded in time; a timeout records ZEROS_ERR_TIMEOUT, raises a CTA
// abort flag and every role leaves its loop; TMEM is released after the last MMA completes.
#include <math.h>

#include <atomic>

#include "zs_common.cuh"
#include "zs_internal.h"
#include "zs_range.cuh"
#include "zs_sm100.cuh"

namespace zs {
namespace {

using namespace sm100;

constexpr int kC = 128;       // tokens per chunk
constexpr int kDV = 32;       // value columns per CTA
constexpr int kThreads = 448;
constexpr uint32_t kTile = 128 * 128;  // one [128 x 64] 16-bit atom tile

// Row coefficients (a, b, g) of a chunk, one block per operand stage.
struct Coef {
  float4 coef[kC];
};

template <int D>
struct Cfg {
  static constexpr int KA = D / 64;              // atom tiles along d
  static constexpr int NSQ = (D == 64) ? 3 : 1;  // q/k stages (with their coefficient blocks)
  static constexpr int NSV = (D == 64) ? 2 : 1;  // scaled value tile stages
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t K_OFF = Q_OFF + NSQ * KA * kTile;
  static constexpr uint32_t V_OFF = K_OFF + NSQ * KA * kTile;
  static constexpr uint32_t VST_OFF = V_OFF + NSV * 2 * kTile;   // raw v slice [128 x 32]
  static constexpr uint32_t SST_OFF = VST_OFF + 128 * 64;
  static constexpr uint32_t RW_OFF = SST_OFF + KA * kTile;       // weight MMA A: [128 x 16] bf16
  static constexpr uint32_t CW_OFF = RW_OFF + kC * 32;           // weight MMA B: [128 x 16] bf16
  static constexpr uint32_t COEF_OFF = CW_OFF + kC * 32;         // Coef [NSQ]
  static constexpr uint32_t PHI_OFF = COEF_OFF + NSQ * (uint32_t)sizeof(Coef);  // float [2][D/2]
  static constexpr uint32_t THETA_OFF = PHI_OFF + 2 * (D / 2) * 4;             // float [D/2]
  static constexpr uint32_t NRM_OFF = THETA_OFF + (D / 2) * 4;   // float2 [2][128] half norms
  static constexpr uint32_t MISC_OFF = NRM_OFF + 2 * kC * 8;
  // output LayerNorm: per-row (mean, M2) of every value slice of the head, two chunk slots
  // (float2 [2][D / kDV][128]), then this slice's gain and bias (float [2][32])
  static constexpr uint32_t LNX_OFF = MISC_OFF + 512;
  static constexpr uint32_t LNW_OFF = LNX_OFF + 2 * (D / kDV) * kC * 8;
  static constexpr uint32_t BYTES = LNW_OFF + 2 * 32 * 4;
  static constexpr uint32_t SMEM = BYTES;  // the base is 1024-byte aligned (checked at entry)
  static constexpr uint32_t TM_A = 0, TM_W = 128, TM_X = 256, TM_ST = 384;
  // S tile (fp16 pairs, A operand of S V): its own 64 columns when d = 64, else the consumed
  // Q K^T columns (then the next Q K^T waits for the S V product)
  static constexpr uint32_t TM_S = (D == 64) ? 448 : 0;
  static_assert(SMEM <= 232448, "shared memory budget of one CTA");
};

constexpr int kMaxNSQ = 3;

struct Misc {
  uint64_t tma_full[kMaxNSQ];
  uint64_t vst_empty;
  uint64_t op_full;      // Vsc of a chunk written
  uint64_t qk_empty[kMaxNSQ];  // Q, K and the coefficients of a stage released
  uint64_t vsc_free[2];  // Vsc of the last chunk of this parity consumed (S V completed)
  uint64_t a_full, a_free, am_full, sst_full, sst_free, st_done, fin;
  uint64_t w_done;       // the weight MMA has read R and C
  uint64_t x_full, x_free;
  uint64_t pobar;        // the operand warps: start of a chunk (rotary base angles written)
  uint64_t nbar;         // the operand warps: half norms of a chunk written
  uint64_t po_sync;      // Q, K, R and C of a chunk written (waited by the MMA thread)
  // coefficients of a chunk written into its stage (waited by the epilogue: one barrier per
  // stage, whose next phase needs the stage's release, which follows the epilogue's read)
  uint64_t cf_full[kMaxNSQ];
  uint64_t ln_full[2];   // output LayerNorm: row statistics of the other value slices landed
  uint32_t tmem;
  int abort;
  int never;  // stays 0: lets the final waits ignore the abort flag
};

static_assert(sizeof(Misc) <= 512, "Misc fits its shared-memory slot");
static_assert(Cfg<64>::NSQ <= kMaxNSQ && Cfg<128>::NSQ <= kMaxNSQ, "one barrier per q/k stage");
static_assert(Cfg<64>::NSV <= 2 && Cfg<128>::NSV <= 2, "vsc_free has one barrier per parity");

struct ChunkParams {
  CUtensorMap tq, tk, tv;  // q, k: box {64, 128, 1} 128B swizzle; v: box {32, 128, 1} 64B swizzle
  FwdArgs a;
};

__device__ __forceinline__ void fail_wait(Misc* ms, int* status) {
  report(status, kErrTimeout);
  ms->abort = 1;
}

__device__ __forceinline__ Coef* coef_block(uint8_t* smem, uint32_t off, int st) {
  return reinterpret_cast<Coef*>(smem + off) + st;
}

// The chunk reference M_c: the running maximum at the chunk's last token.
__device__ __forceinline__ float chunk_ref(const float4* __restrict__ scal, int c, int N) {
  return __ldg(&scal[min(N, (c + 1) * kC) - 1].y);
}

// Before the Vsc tile of chunk c is written: the S V product of chunk c - NS (same stage) has
// completed.  One barrier per chunk parity, waited in consecutive phases.
template <int D>
__device__ __forceinline__ bool vsc_wait(Misc* ms, int c) {
  constexpr int NS = Cfg<D>::NSV;
  if (c < NS) return true;
  return mbar_wait_warp(&ms->vsc_free[(c - NS) & 1], (uint32_t)((c - NS) >> 1) & 1u, &ms->abort);
}

// Vsc row r, 16-byte pieces x0, x0 + 1 of the value row, fp16: the value itself (exact for bf16
// values in the fp16 range) to columns 8 x .. 8 x + 7 of atom 0, then the scaled parts:
// atom 0 = [v | e v], atom 1 = [s' v | k v], from the row's column scalars (e, s', k) (s'
// already carries G's 2^-ks).  Returns the largest |v| as bf16 pairs.
__device__ __forceinline__ uint32_t build_vsc_half(uint8_t* vt, const uint8_t* vst, int r,
                                                   int x0, float ce, float cs1, float ck) {
  const float2 ce2 = make_float2(ce, ce), cs2 = make_float2(cs1, cs1), ck2 = make_float2(ck, ck);
  uint32_t vmax = 0u;
#pragma unroll
  for (int x = x0; x < x0 + 2; ++x) {
    const uint4 wv = *reinterpret_cast<const uint4*>(vst + sw64_off(r, x));
    const uint32_t pv[4] = {wv.x, wv.y, wv.z, wv.w};
    uint32_t ph[4], pe[4], ps[4], pk[4];
#pragma unroll
    for (int y = 0; y < 4; ++y) {
      float2 v2;
      unpack_bf16x2(pv[y], v2.x, v2.y);
      vmax = bf16x2_absmax(vmax, pv[y]);
      const float2 e2 = __fmul2_rn(ce2, v2), s2 = __fmul2_rn(cs2, v2), k2 = __fmul2_rn(ck2, v2);
      ph[y] = pack_f16x2(v2.x, v2.y);
      pe[y] = pack_f16x2(e2.x, e2.y);
      ps[y] = pack_f16x2(s2.x, s2.y);
      pk[y] = pack_f16x2(k2.x, k2.y);
    }
    *reinterpret_cast<uint4*>(vt + sw128_off(r, x)) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
    *reinterpret_cast<uint4*>(vt + sw128_off(r, 4 + x)) = make_uint4(pe[0], pe[1], pe[2], pe[3]);
    *reinterpret_cast<uint4*>(vt + kTile + sw128_off(r, x)) = make_uint4(ps[0], ps[1], ps[2], ps[3]);
    *reinterpret_cast<uint4*>(vt + kTile + sw128_off(r, 4 + x)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
  return vmax;
}

// bf16 values from 45056 up (and inf, NaN) are beyond what the fp16 operands hold once rotated
// (a rotation grows an element by up to sqrt 2; fp16 ends at 65504).
__device__ __forceinline__ bool beyond_f16(uint32_t bf16x2_max, uint32_t limit) {
  return (bf16x2_max & 0xffffu) >= limit || (bf16x2_max >> 16) >= limit;
}
constexpr uint32_t kBf16RotLimit = 0x4730u;  // 45056
constexpr uint32_t kBf16Limit = 0x4780u;     // 65536

// ============================================================================ T: TMA producer
template <int D>
__device__ void role_tma(const ChunkParams& p, uint8_t* smem, Misc* ms, int bh, int nch) {
  using CF = Cfg<D>;
  const uint32_t base = smem_u32(smem);
  const int j0 = blockIdx.y * kDV;
  constexpr uint32_t qk_bytes = 2 * CF::KA * kTile, v_bytes = 128 * 64;
  tma_prefetch_desc(&p.tq);
  tma_prefetch_desc(&p.tk);
  tma_prefetch_desc(&p.tv);
  for (int c = 0; c < nch; ++c) {
    const int st = c % CF::NSQ;
    if (c >= CF::NSQ) {
      // the chunk's tiles start towards L2 while the stage is still in use
#pragma unroll
      for (int at = 0; at < CF::KA; ++at) {
        tma_prefetch_3d(&p.tq, 64 * at, c * kC, bh);
        tma_prefetch_3d(&p.tk, 64 * at, c * kC, bh);
      }
      tma_prefetch_3d(&p.tv, j0, c * kC, bh);
      if (!mbar_wait(&ms->qk_empty[st], ((c / CF::NSQ) - 1) & 1, &ms->abort)) {
        fail_wait(ms, p.a.status);
        return;
      }
    }
    uint64_t* tf = &ms->tma_full[st];
    mbar_arrive_expect_tx(tf, qk_bytes + v_bytes);
    const uint32_t qt = base + CF::Q_OFF + st * CF::KA * kTile;
    const uint32_t kt = base + CF::K_OFF + st * CF::KA * kTile;
#pragma unroll
    for (int at = 0; at < CF::KA; ++at) {
      tma_load_3d(qt + at * kTile, &p.tq, 64 * at, c * kC, bh, tf);
      tma_load_3d(kt + at * kTile, &p.tk, 64 * at, c * kC, bh, tf);
    }
    // the raw value slice has one buffer, released by the operand warps once copied
    if (c >= 1 && !mbar_wait(&ms->vst_empty, (c - 1) & 1, &ms->abort)) {
      fail_wait(ms, p.a.status);
      return;
    }
    tma_load_3d(base + CF::VST_OFF, &p.tv, j0, c * kC, bh, tf);
  }
}

// ============================================================================ O: operands
// Rotates (RoPE) pair group g (pairs 8g .. 8g+7 with partners + D/2) of row r of a
// 128B-swizzled bf16 tile in place, as fp16 (converted without rotation when rope is off),
// accumulates the row's squared norm into ss (two partial sums) and the largest |x| (bf16
// pairs) into amax.  cs[k] = (cos, sin) of pair 8g + k.
template <int D>
__device__ __forceinline__ void rotate_group(uint8_t* tile, int r, int g, bool rope,
                                             const float2 (&cs)[8], float2& ss, uint32_t& amax) {
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
    amax = bf16x2_absmax(bf16x2_absmax(amax, wl[k]), wh[k]);
    ss = __ffma2_rn(xa, xa, ss);
    ss = __ffma2_rn(xb, xb, ss);
    if (rope) {
      // pair (a, b) -> (a c - b s, a s + b c), one pair per component of the f32x2 ops
      const float2 c2 = make_float2(cs[2 * k].x, cs[2 * k + 1].x);
      const float2 s2 = make_float2(cs[2 * k].y, cs[2 * k + 1].y);
      const float2 na = __ffma2_rn(xa, c2, __fmul2_rn(make_float2(-xb.x, -xb.y), s2));
      const float2 nb = __ffma2_rn(xa, s2, __fmul2_rn(xb, c2));
      oa[k] = pack_f16x2(na.x, na.y);
      ob[k] = pack_f16x2(nb.x, nb.y);
    } else {
      oa[k] = pack_f16x2(xa.x, xa.y);
      ob[k] = pack_f16x2(xb.x, xb.y);
    }
  }
  *pa = make_uint4(oa[0], oa[1], oa[2], oa[3]);
  *pb = make_uint4(ob[0], ob[1], ob[2], ob[3]);
}

// Per chunk: rotation of this half's rotary pairs of q and k, the row's norms (halves summed
// through shared memory), then hf = 0: row coefficients (a, b, g) and the row weight operand;
// hf = 1: the column weight operand; both: half of the row's Vsc.
template <int D>
__device__ void role_operands(const FwdArgs& a, uint8_t* smem, Misc* ms, size_t row0, int nch) {
  using CF = Cfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hf = warp >> 2;         // which half of the row's work
  const int r = 32 * (warp & 3) + lane;  // token row inside the chunk, 0..127
  const int N = a.N;
  const float4* __restrict__ scal = a.scal + row0;
  const int ks = s_exp(a, blockIdx.x);          // G is carried with s 2^-ks
  const float sinv = pow2f(-ks);
  const float smax = seq_smax(a, blockIdx.x);   // the sequence's largest |s|
  float* phi = reinterpret_cast<float*>(smem + CF::PHI_OFF);      // [2][D/2]
  float* theta = reinterpret_cast<float*>(smem + CF::THETA_OFF);  // [D/2]
  float2* nrm = reinterpret_cast<float2*>(smem + CF::NRM_OFF);    // [2][128] (|q|^2, |k|^2)
  const double two_pi = 6.283185307179586476925286766559;
  const int pj = threadIdx.x;  // rotary pair owned for the tables (threads 0 .. D/2 - 1)
  const bool owns_pair = a.rope && pj < D / 2;
  double theta_d = 0.0;
  if (owns_pair) {
    theta_d = pow((double)a.rope_base, -2.0 * (double)pj / (double)D);
    theta[pj] = (float)theta_d;
  }

  // rotary base angle of chunk cc per pair, reduced modulo 2 pi in fp64; token r of the chunk
  // then uses phi_j + r theta_j.  Written one chunk ahead (double buffer, pobar orders it).
  auto put_phi = [&](int cc, int slot) {
    if (owns_pair) {
      const double ang = (double)(cc * kC) * theta_d;
      phi[slot * (D / 2) + pj] = (float)(ang - rint(ang * (1.0 / two_pi)) * two_pi);
    }
  };
  // inputs of chunk cc that are loaded one chunk ahead (their latency is hidden): the token's
  // scalars, the chunk reference and the gate logits (x0: optional zero-order gate, -inf when
  // absent, so that its sigmoid is 0)
  struct Ahead {
    float4 sc;
    float M, Mp, x1, xh, x0;  // Mp: the running maximum at the token before the chunk
  };
  auto load_ahead = [&](int cc) {
    Ahead o{make_float4(0.f, 0.f, 0.f, 0.f), 0.0f, 0.0f, 0.0f, 0.0f, -INFINITY};
    if (cc < nch) {
      o.M = chunk_ref(scal, cc, N);
      if (cc > 0) o.Mp = __ldg(&scal[cc * kC - 1].y);
      const int i = cc * kC + r;
      if (i < N) {
        o.sc = __ldg(scal + i);
        if (hf == 0) {
          o.x1 = __ldg(a.g1 + row0 + i);
          o.xh = __ldg(a.gh + row0 + i);
          if (a.g0) o.x0 = __ldg(a.g0 + row0 + i);
        }
      }
    }
    return o;
  };
  put_phi(0, 0);
  Ahead cur = load_ahead(0), nxt{};

  for (int c = 0; c < nch; ++c) {
    const int st = c % CF::NSQ;
    const int i = c * kC + r;
    const bool valid = i < N;
    mbar_arrive(&ms->pobar);
    if (!mbar_wait_warp(&ms->pobar, c & 1, &ms->abort)) {
      fail_wait(ms, a.status);
      return;
    }
    if (!mbar_wait_warp(&ms->tma_full[st], (uint32_t)(c / CF::NSQ) & 1u, &ms->abort)) {
      fail_wait(ms, a.status);
      return;
    }
    uint8_t* qt = smem + CF::Q_OFF + st * CF::KA * kTile;
    uint8_t* kt = smem + CF::K_OFF + st * CF::KA * kTile;
    uint8_t* vt = smem + CF::V_OFF + (c % CF::NSV) * 2 * kTile;
    nxt = load_ahead(c + 1);
    // ---- rotate this half's pair groups of q and k in place (TMA tiles), half norms ----
    const bool rot = a.rope != 0 && valid;
    float2 qq2 = make_float2(0.0f, 0.0f), kk2 = make_float2(0.0f, 0.0f);
    uint32_t amax = 0u;  // the row's largest |q|, |k| elements (bf16 pairs)
    {
      const float* ph = phi + (c & 1) * (D / 2);
      const float rf = (float)r;
      constexpr int GH = D / 32;  // pair groups per half
#pragma unroll
      for (int gg = 0; gg < GH; ++gg) {
        const int g = hf * GH + gg;
        float2 cs[8];
        if (rot) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float sn, cn;
            __sincosf(__fmaf_rn(rf, theta[8 * g + k], ph[8 * g + k]), &sn, &cn);
            cs[k] = make_float2(cn, sn);
          }
        }
        rotate_group<D>(qt, r, g, rot, cs, qq2, amax);
        rotate_group<D>(kt, r, g, rot, cs, kk2, amax);
      }
    }
    if (beyond_f16(amax, kBf16RotLimit)) report(a.status, kErrRange);
    nrm[hf * kC + r] = make_float2(__fadd_rn(qq2.x, qq2.y), __fadd_rn(kk2.x, kk2.y));
    mbar_arrive(&ms->nbar);
    if (!mbar_wait_warp(&ms->nbar, c & 1, &ms->abort)) {
      fail_wait(ms, a.status);
      return;
    }
    const float2 n0 = nrm[r], n1 = nrm[kC + r];
    const float qq = __fadd_rn(n0.x, n1.x), kq = __fadd_rn(n0.y, n1.y);
    // column scalars and row coefficients (these feed 16-bit / fp32 products, not the scalar
    // contract: fast exp, reciprocal square root and division are accurate enough here)
    const float s = cur.sc.x, m = cur.sc.y, Et = cur.sc.z, P = cur.sc.w, M = cur.M;
    const float kap = rsqrtf(fmaxf(kq, 1e-24f));
    float ce = 0.0f, cs1 = 0.0f, ck = 0.0f;
    float4 cf = make_float4(0.f, 0.f, 0.f, 0.f);  // (a, b, g) of the weight operand
    // the output's coefficients of X_F, X_G, X_H (scaled for the fp16 state copy: 2^kb, and
    // 2^ks for G; X_F's copy is referenced to the running maximum before the chunk) and the
    // row's S scale 2^kr
    float4 co = make_float4(0.f, 0.f, 0.f, 1.f);
    if (valid) {
      ce = __fmul_rn(__expf(__fsub_rn(s, M)), kap);
      cs1 = __fmul_rn(s, kap);
      ck = kap;
      if (hf == 0) {
        const float rho = rsqrtf(fmaxf(qq, 1e-24f));
        const float sig1 = __fdividef(1.0f, 1.0f + __expf(-cur.x1));
        const float sigh = __fdividef(1.0f, 1.0f + __expf(-cur.xh));
        const float rt = __fdividef(1.0f, (float)(i + 1));
        const float b0c = (sig1 - sigh) * rt;
        const float ahat = __fdividef(sigh, Et) * __expf(M - m);
        float g0c = -(b0c * P * rt + sigh * rt);
        if (a.g0) g0c += __fdividef(1.0f, 1.0f + __expf(-cur.x0)) * rt;  // zero-order
        cf.x = rho * ahat;
        cf.y = rho * b0c;
        cf.z = rho * g0c;
        if (!isfinite(cf.x)) report(a.status, kErrRange);
        const float kb2 = pow2f(state_exp(c, kC));
        co.x = c > 0 ? rho * __fdividef(sigh, Et) * __expf(cur.Mp - m) * kb2 : 0.0f;
        co.y = cf.y * kb2 * pow2f(ks);
        co.z = cf.z * kb2;
        // a e_i over the row's keys i <= t is at most sigma^h / E~ (e^{s_i - m_t} <= 1)
        co.w = pow2f(row_exp(__fdividef(sigh, Et) + fabsf(b0c) * smax + fabsf(g0c)));
      } else if (!isfinite(ce)) {
        report(a.status, kErrRange);
      }
    }
    if (hf == 0) {
      coef_block(smem, CF::COEF_OFF, st)->coef[r] = co;
      mbar_arrive(&ms->cf_full[st]);
    }
    // Weight operands: W_{t,i} = a_t e_i + b_t s'_i + g_t k_i is formed by one K = 16 MMA of
    // the row vector [a a' a a' b b' b b' g g' g g' 0 0 0 0] (hi and lo bf16 parts,
    // x = x + x') and the column vector [e e' e e' s s' s s' k k' k k' 0 0 0 0] paired as
    // (hi hi, hi lo, lo hi, lo lo): every product is exact in fp32, the representation error
    // is about 2^-17 of each term, so the nearly cancelling sum keeps fp32-level accuracy.
    // The buffer is single: the previous chunk's weight MMA must have completed.
    if (c >= 1 && !mbar_wait_warp(&ms->w_done, (c - 1) & 1, &ms->abort)) {
      fail_wait(ms, a.status);
      return;
    }
    {
      const float x0 = hf == 0 ? cf.x : ce, x1 = hf == 0 ? cf.y : cs1, x2 = hf == 0 ? cf.z : ck;
      const float h0 = __bfloat162float(__float2bfloat16_rn(x0));
      const float h1 = __bfloat162float(__float2bfloat16_rn(x1));
      const float h2 = __bfloat162float(__float2bfloat16_rn(x2));
      const float l0 = __fsub_rn(x0, h0), l1 = __fsub_rn(x1, h1), l2 = __fsub_rn(x2, h2);
      if (hf == 0) {
        uint8_t* rw = smem + CF::RW_OFF;
        *reinterpret_cast<uint4*>(rw + sw32_off(r, 0)) =
            make_uint4(pack_bf16x2(h0, h0), pack_bf16x2(l0, l0), pack_bf16x2(h1, h1),
                       pack_bf16x2(l1, l1));
        *reinterpret_cast<uint4*>(rw + sw32_off(r, 1)) =
            make_uint4(pack_bf16x2(h2, h2), pack_bf16x2(l2, l2), 0u, 0u);
      } else {
        uint8_t* cw = smem + CF::CW_OFF;
        *reinterpret_cast<uint4*>(cw + sw32_off(r, 0)) =
            make_uint4(pack_bf16x2(h0, l0), pack_bf16x2(h0, l0), pack_bf16x2(h1, l1),
                       pack_bf16x2(h1, l1));
        *reinterpret_cast<uint4*>(cw + sw32_off(r, 1)) =
            make_uint4(pack_bf16x2(h2, l2), pack_bf16x2(h2, l2), 0u, 0u);
      }
    }
    // Q, K, R, C and the coefficients are complete: the MMA may start
    fence_proxy_async_smem();
    mbar_arrive(&ms->po_sync);
    // half of the value row: raw bf16 words to the Vsc tile (once the stage's previous Vsc was
    // consumed), the staging buffer handed back, then the scaled parts
    if (!vsc_wait<D>(ms, c)) {
      fail_wait(ms, a.status);
      return;
    }
    const uint32_t vmax = build_vsc_half(vt, smem + CF::VST_OFF, r, 2 * hf, ce, cs1 * sinv, ck);
    if (beyond_f16(vmax, kBf16Limit)) report(a.status, kErrRange);
    mbar_arrive(&ms->vst_empty);
    fence_proxy_async_smem();
    mbar_arrive(&ms->op_full);
    if (c + 1 < nch) put_phi(c + 1, (c + 1) & 1);
    cur = nxt;
  }
}

// ============================================================================ M: MMA issue
// Per chunk c, in issue order (each group waits only for what it reads or overwrites):
//   A = Q K^T and W = R C^T                 (Q, K, R, C written; previous S tile formed)
//                                                                         -> a_full, w_done
//   state += Vsc^T K                        (state copied to the B tile, F~ rescaled)  -> st_done
//   X[:, 0:96] = Q [F~ | G | H] (c >= 1)    (previous outputs read from X)
//                                                                      -> sst_free, qk_empty
//   X[:, 96:128] = S V                      (this chunk's S tile formed)   -> x_full, vsc_free
// qk_empty follows the Q [F|G|H] product (the S V product for the first chunk).  The epilogue
// reads a chunk's coefficients before it frees X of the previous chunk, which the Q [F|G|H]
// product waits for.
template <int D>
__device__ void role_mma(const FwdArgs& a, uint8_t* smem, Misc* ms, int nch) {
  using CF = Cfg<D>;
  const bool leader = elect_one();
  const uint32_t base = smem_u32(smem);
  const uint32_t tm = ms->tmem;
  const uint32_t tA = tm + CF::TM_A, tW = tm + CF::TM_W, tX = tm + CF::TM_X, tS = tm + CF::TM_ST;
  constexpr uint32_t id_qk = idesc_f16_f32(128, 128, false, false);    // Q K^T
  constexpr uint32_t id_w = idesc_bf16_f32(128, 128, false, false);    // R C^T (hi/lo bf16)
  constexpr uint32_t id_qs = idesc_f16_f32(128, 96, false, false);     // Q [F|G|H]
  constexpr uint32_t id_sv = idesc_f16_f32(128, 32, false, true);      // S V
  constexpr uint32_t id_st = idesc_f16_f32(128, D, true, true);        // Vsc^T K
  const uint64_t d_rw = sw32_desc(base + CF::RW_OFF), d_cw = sw32_desc(base + CF::CW_OFF);
  bool ok = true;
  // descriptors: the start address field is (address >> 4), and every tile lies below 256 KB,
  // so the descriptor of base + off is the base's descriptor + off / 16
  const uint64_t dq0 = sw128_desc(base + CF::Q_OFF, 16, 1024);
  const uint64_t dk0 = sw128_desc(base + CF::K_OFF, 16, 1024);
  const uint64_t dkm0 = sw128_desc(base + CF::K_OFF, kTile, 1024);   // K as MN-major B
  const uint64_t dv0 = sw128_desc(base + CF::V_OFF, kTile, 1024);
  const uint64_t dsst = sw128_desc(base + CF::SST_OFF + 32 * 128, 16, 1024);
  for (int c = 0; c < nch && ok; ++c) {
    const int st = c % CF::NSQ;
    const uint32_t ph = (uint32_t)c & 1u;
    const uint64_t sq = (uint64_t)((st * CF::KA * kTile) >> 4);
    const uint64_t sv = (uint64_t)(((c % CF::NSV) * 2 * kTile) >> 4);
    ok = mbar_wait_warp(&ms->po_sync, ph, &ms->abort);
    if (ok && c >= 1) ok = mbar_wait_warp(&ms->a_free, (c - 1) & 1, &ms->abort);
    // the S tile shares the Q K^T columns: the previous S V product must have read it
    if (CF::TM_S == CF::TM_A && ok && c >= 1)
      ok = mbar_wait_warp(&ms->x_full, (c - 1) & 1, &ms->abort);
    if (!ok) break;
    tc_fence_after();
    // ---- A = Q K^T (K = d); W = R C^T (K = 16) ----
    if (leader) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = (uint64_t)(((kk / 4) * kTile + (kk % 4) * 32) >> 4);
        mma_f16kind(tA, dq0 + sq + off, dk0 + sq + off, id_qk, kk > 0);
      }
      mma_f16kind(tW, d_rw, d_cw, id_w, 0u);
      mma_commit(&ms->a_full);
      mma_commit(&ms->w_done);
    }
    __syncwarp();
    // ---- state^T += Vsc^T K (M = 128 value rows, N = d, K = chunk tokens) ----
    if (c >= 1 && !mbar_wait_warp(&ms->sst_full, (c - 1) & 1, &ms->abort)) { ok = false; break; }
    if (!mbar_wait_warp(&ms->op_full, ph, &ms->abort)) { ok = false; break; }
    tc_fence_after();
    if (leader) {
#pragma unroll
      for (int kk = 0; kk < kC / 16; ++kk) {
        const uint64_t off = (uint64_t)((kk * 2048) >> 4);
        mma_f16kind(tS, dv0 + sv + off, dkm0 + sq + off, id_st, (c > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(&ms->st_done);
    }
    __syncwarp();
    // ---- X[:, 0:96] = Q [F~ | G | H] (state of the previous chunks, B tile rows 32..127) ----
    if (c >= 1) {
      if (!mbar_wait_warp(&ms->x_free, (c - 1) & 1, &ms->abort)) { ok = false; break; }
      tc_fence_after();
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk / 4) * kTile + (kk % 4) * 32) >> 4);
          mma_f16kind(tX, dq0 + sq + off, dsst + off, id_qs, kk > 0);
        }
        mma_commit(&ms->sst_free);
        mma_commit(&ms->qk_empty[st]);  // Q, K and the coefficients of this chunk: not read again
      }
      __syncwarp();
    }
    // ---- X[:, 96:128] = S V ----
    if (!mbar_wait_warp(&ms->am_full, c & 1, &ms->abort)) { ok = false; break; }
    tc_fence_after();
    if (leader) {
#pragma unroll
      for (int kk = 0; kk < kC / 16; ++kk) {
        const uint64_t boff = (uint64_t)((kk * 2048) >> 4);  // MN-major B, 16 token rows/step
        mma_f16kind_ts(tX + 96, tm + CF::TM_S + kk * 8, dv0 + sv + boff, id_sv, kk > 0);
      }
      mma_commit(&ms->x_full);
      if (c == 0) mma_commit(&ms->qk_empty[st]);  // no Q [F|G|H] product: after S was read
      mma_commit(&ms->vsc_free[c & 1]);
    }
    __syncwarp();
  }
  if (leader) {
    if (!ok) fail_wait(ms, a.status);
    mma_commit(&ms->fin);
  }
  __syncwarp();
}

// ============================================================================ E: epilogue
// Per chunk c: the S tile (A o W, masked, bf16), the state after chunk c as the bf16 B tile of
// chunk c+1 (F~ rescaled to M_{c+1}), then the output rows of chunk c.  The chunk references
// come from the scalar pass, so the state copy waits only for the state update.
template <int D, bool LN>
__device__ void role_epilogue(const FwdArgs& a, uint8_t* smem, Misc* ms, int bh, size_t row0,
                              int nch) {
  using CF = Cfg<D>;
  const int wq = (threadIdx.x >> 5) & 3;          // TMEM lane quadrant of this warp
  const int t = wq * 32 + (threadIdx.x & 31);     // TMEM lane = token row / state row
  const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
  const uint32_t tm = ms->tmem + lane_off;
  const uint32_t base = smem_u32(smem);
  const int j0 = blockIdx.y * kDV;
  const int N = a.N;
  const float4* __restrict__ scal = a.scal + row0;
  __nv_bfloat16* __restrict__ out = static_cast<__nv_bfloat16*>(a.out) + row0 * D;
  bool ok = true;
  // (a, b, g) of row t of the current chunk: read while the previous chunk is in flight (before
  // X of that chunk is freed), since the coefficient block is released with the chunk's Q, K
  float4 cf = make_float4(0.f, 0.f, 0.f, 0.f);
  float M_cur = 0.0f;
  if (nch > 0) {
    M_cur = chunk_ref(scal, 0, N);
    ok = mbar_wait_warp(&ms->cf_full[0], 0, &ms->abort);
    if (ok) cf = coef_block(smem, CF::COEF_OFF, 0)->coef[t];
  }
  for (int c = 0; c < nch && ok; ++c) {
    float4 cf_next = make_float4(0.f, 0.f, 0.f, 0.f);
    const float M_next = c + 1 < nch ? chunk_ref(scal, c + 1, N) : 0.0f;
    // ---- S = [i <= t] (Q K^T) o W 2^kr_t, fp32 product then fp16 (rows t, K = token i) ----
    ok = mbar_wait_warp(&ms->a_full, c & 1, &ms->abort);
    if (!ok) break;
    tc_fence_after();
    // 16-column piece h of S (columns 16h..16h+15) goes to the 8 packed columns 8h.. of the S
    // tile; pieces are double-buffered (the load of piece h+1 is in flight while piece h is
    // formed).  With the S tile on the Q K^T columns, every column written was read before.
    {
      const int npiece = 2 * (wq + 1);  // pieces holding entries i <= t for some row of the warp
      uint32_t ra0[16], rw0[16], ra1[16], rw1[16];
      auto piece = [&](int h, uint32_t (&ra)[16], uint32_t (&rw)[16]) {
        uint32_t pw[8];
#pragma unroll
        for (int y = 0; y < 8; ++y) {
          float2 val = __fmul2_rn(make_float2(__uint_as_float(ra[2 * y]), __uint_as_float(ra[2 * y + 1])),
                                  make_float2(__uint_as_float(rw[2 * y]), __uint_as_float(rw[2 * y + 1])));
          val = __fmul2_rn(val, make_float2(cf.w, cf.w));  // the row's 2^kr
          const int col = 16 * h + 2 * y;
          if ((h >> 1) == wq) {  // diagonal block: keep i <= t only
            if (col > t) val.x = 0.0f;
            if (col + 1 > t) val.y = 0.0f;
          }
          pw[y] = pack_f16x2(val.x, val.y);
        }
        tmem_st8_nowait(tm + CF::TM_S + 8 * h, pw);
      };
      tmem_ld16_nowait(tm + CF::TM_A, ra0);
      tmem_ld16_nowait(tm + CF::TM_W, rw0);
#pragma unroll 1
      for (int h = 0; h < npiece; h += 2) {
        tmem_wait_ld();
        reg_fence(ra0);
        reg_fence(rw0);
        tmem_ld16_nowait(tm + CF::TM_A + 16 * (h + 1), ra1);
        tmem_ld16_nowait(tm + CF::TM_W + 16 * (h + 1), rw1);
        piece(h, ra0, rw0);
        tmem_wait_ld();
        reg_fence(ra1);
        reg_fence(rw1);
        if (h + 2 < npiece) {
          tmem_ld16_nowait(tm + CF::TM_A + 16 * (h + 2), ra0);
          tmem_ld16_nowait(tm + CF::TM_W + 16 * (h + 2), rw0);
        }
        piece(h + 1, ra1, rw1);
      }
    }
    {
      // blocks after every row of this warp are zero
      uint32_t zw[16];
#pragma unroll
      for (int y = 0; y < 16; ++y) zw[y] = 0u;
#pragma unroll 1
      for (int cb = wq + 1; cb < 4; ++cb) tmem_st16_nowait(tm + CF::TM_S + cb * 16, zw);
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&ms->a_free);
    mbar_arrive(&ms->am_full);
    // ---- state after chunk c -> fp16 B operand rows 32..127 of chunk c+1 (times 2^-kb, F~ at
    //      its reference M_cur), F~ in TMEM rescaled to M_next for the next update ----
    if (c + 1 < nch) {
      ok = mbar_wait_warp(&ms->st_done, c & 1, &ms->abort);
      if (ok && c >= 1) ok = mbar_wait_warp(&ms->sst_free, (c - 1) & 1, &ms->abort);
      if (!ok) break;
      tc_fence_after();
      if (wq >= 1) {
        const bool rescale = (wq == 1) && (M_next > M_cur);
        const float fac = rescale ? expf(__fsub_rn(M_cur, M_next)) : 1.0f;
        const float2 sc2 = make_float2(pow2f(-state_exp(c + 1, kC)), pow2f(-state_exp(c + 1, kC)));
        const uint32_t sst = base + CF::SST_OFF;
        // 32 state columns per round: two 16-column loads, one wait
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t rr[2][16];
#pragma unroll
          for (int q = 0; q < 2; ++q) tmem_ld16_nowait(tm + CF::TM_ST + c0 + 16 * q, rr[q]);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 2; ++q) reg_fence(rr[q]);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              const uint32_t* w8 = rr[q] + 8 * x;
              uint32_t pk[4];
#pragma unroll
              for (int y = 0; y < 4; ++y) {
                const float2 f = __fmul2_rn(make_float2(__uint_as_float(w8[2 * y]),
                                                        __uint_as_float(w8[2 * y + 1])), sc2);
                pk[y] = pack_f16x2(f.x, f.y);
              }
              const int col0 = c0 + 16 * q + 8 * x;
              sts128(sst + (col0 / 64) * kTile + sw128_off(t, (col0 % 64) / 8),
                     make_uint4(pk[0], pk[1], pk[2], pk[3]));
            }
          }
          if (rescale) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
#pragma unroll
              for (int y = 0; y < 16; ++y)
                rr[q][y] = __float_as_uint(__fmul_rn(__uint_as_float(rr[q][y]), fac));
              tmem_st16_nowait(tm + CF::TM_ST + c0 + 16 * q, rr[q]);
            }
            tmem_wait_st();
          }
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(&ms->sst_full);
    }
    // ---- o = X_SV + a X_F + b X_G + g X_H for the rows of chunk c (two 16-column halves) ----
    ok = mbar_wait_warp(&ms->x_full, c & 1, &ms->abort);
    if (!ok) break;
    tc_fence_after();
    const int i = c * kC + t;
    uint4* dst = reinterpret_cast<uint4*>(out + (size_t)i * D + j0);
    // the 16 outputs of half hf of row t (fp32 bit patterns)
    auto out_half = [&](int hf, uint32_t (&rsv)[16]) {
      const uint32_t tx = tm + CF::TM_X + hf * 16;
      uint32_t rx[16];
      tmem_ld16_nowait(tx + 96, rsv);
      if (c >= 1) tmem_ld16_nowait(tx + 0, rx);
      tmem_wait_ld();
      reg_fence(rsv);
      const float rinv = __frcp_rn(cf.w);  // S V carries the row's 2^kr
#pragma unroll
      for (int j = 0; j < 16; ++j) rsv[j] = __float_as_uint(__uint_as_float(rsv[j]) * rinv);
      if (c >= 1) {
        reg_fence(rx);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          rsv[j] = __float_as_uint(__fmaf_rn(cf.x, __uint_as_float(rx[j]), __uint_as_float(rsv[j])));
        uint32_t ry[16];
        tmem_ld16_nowait(tx + 32, rx);
        tmem_ld16_nowait(tx + 64, ry);
        tmem_wait_ld();
        reg_fence(rx);
        reg_fence(ry);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          rsv[j] = __float_as_uint(__fmaf_rn(cf.z, __uint_as_float(ry[j]),
                                             __fmaf_rn(cf.y, __uint_as_float(rx[j]),
                                                       __uint_as_float(rsv[j]))));
      }
    };
    float ln_mean = 0.0f, ln_rstd = 1.0f;
    if constexpr (LN) {
      // Output LayerNorm over the head's d columns, split over the D / 32 value-slice CTAs of
      // the cluster: each publishes its rows' (mean, M2) over its 32 columns (shifted sums),
      // the statistics are merged (pairwise moment update), and the
      // outputs are recomputed from TMEM (X stays allocated until x_free) and normalised.
      constexpr int NSL = D / kDV;
      float sh = 0.0f, s1 = 0.0f, s2 = 0.0f;
#pragma unroll 1
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t rsv[16];
        out_half(hf, rsv);
        if (hf == 0) sh = __uint_as_float(rsv[0]);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float dv = __uint_as_float(rsv[j]) - sh;
          s1 += dv;
          s2 = __fmaf_rn(dv, dv, s2);
        }
      }
      const float lmean = sh + s1 * (1.0f / kDV);
      const float lm2 = fmaxf(s2 - s1 * s1 * (1.0f / kDV), 0.0f);
      const int me = blockIdx.y;
      float2* lnx = reinterpret_cast<float2*>(smem + CF::LNX_OFF);
      const uint32_t slot = smem_u32(&lnx[((c & 1) * NSL + me) * kC + t]);
#pragma unroll
      for (int r = 1; r < NSL; ++r) st_cluster_f32x2(mapa(slot, (me + r) % NSL), lmean, lm2);
      __syncwarp();
      if ((threadIdx.x & 31) == 0) {
#pragma unroll
        for (int r = 1; r < NSL; ++r)
          mbar_arrive_remote(mapa(smem_u32(&ms->ln_full[c & 1]), (me + r) % NSL));
      }
      ok = mbar_wait_cl_warp(&ms->ln_full[c & 1], (uint32_t)(c >> 1) & 1u, &ms->abort);
      if (!ok) break;
      float cnt = (float)kDV, mean = lmean, m2 = lm2;  // merged over the slices
#pragma unroll
      for (int r = 1; r < NSL; ++r) {
        const float2 o = lnx[((c & 1) * NSL + (me + r) % NSL) * kC + t];
        moments_merge(cnt, mean, m2, (float)kDV, o.x, o.y);
      }
      ln_mean = mean;
      ln_rstd = rsqrtf(m2 * (1.0f / D) + a.ln_eps);
    }
#pragma unroll 1
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t rsv[16];
      out_half(hf, rsv);
      if constexpr (LN) {
        const float* lw = reinterpret_cast<const float*>(smem + CF::LNW_OFF);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float y = (__uint_as_float(rsv[j]) - ln_mean) * ln_rstd;
          rsv[j] = __float_as_uint(__fmaf_rn(y, lw[16 * hf + j], lw[32 + 16 * hf + j]));
        }
      }
      uint32_t ob[8];  // the half's 16 outputs as bf16 pairs
#pragma unroll
      for (int j = 0; j < 8; ++j)
        ob[j] = pack_bf16x2(__uint_as_float(rsv[2 * j]), __uint_as_float(rsv[2 * j + 1]));
      if (hf == 1) {
        // the next chunk's coefficients, before its coefficient block can be released
        if (c + 1 < nch) {
          const int sn = (c + 1) % CF::NSQ;
          ok = mbar_wait_warp(&ms->cf_full[sn], (uint32_t)((c + 1) / CF::NSQ) & 1u, &ms->abort);
          if (!ok) break;
          cf_next = coef_block(smem, CF::COEF_OFF, sn)->coef[t];
        }
        tc_fence_before();
        mbar_arrive(&ms->x_free);
      }
      if (i < N) {
        dst[2 * hf + 0] = make_uint4(ob[0], ob[1], ob[2], ob[3]);
        dst[2 * hf + 1] = make_uint4(ob[4], ob[5], ob[6], ob[7]);
      }
    }
    if (!ok) break;
    cf = cf_next;
    M_cur = M_next;
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
      const float gs = wq == 2 ? pow2f(s_exp(a, bh)) : 1.0f;  // G was carried with s 2^-ks
#pragma unroll
      for (int cb = 0; cb < D / 32; ++cb) {
        float v[32];
        tmem_ld32(tm + CF::TM_ST + cb * 32, v);
#pragma unroll
        for (int y = 0; y < 32; ++y) rec[off + (cb * 32 + y) * D + j0 + j] = v[y] * gs;
      }
    }
  }
}

// ============================================================================ kernel
template <int D, bool LN>
__global__ void __launch_bounds__(kThreads, 1) chunk_kernel(const __grid_constant__ ChunkParams p) {
  using CF = Cfg<D>;
  const FwdArgs& a = p.a;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (smem_u32(smem) & 1023u) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) report(a.status, kErrUnsupported);
    return;
  }
  Misc* ms = reinterpret_cast<Misc*>(smem + CF::MISC_OFF);
  const int warp = threadIdx.x >> 5;
  const int bh = blockIdx.x;
  const size_t row0 = (size_t)bh * a.N;
  const int nch = (a.N + kC - 1) / kC;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) mbar_init(&ms->vsc_free[i], 1);
    for (int i = 0; i < kMaxNSQ; ++i) {
      mbar_init(&ms->tma_full[i], 1);
      mbar_init(&ms->qk_empty[i], 1);
      mbar_init(&ms->cf_full[i], 128);
    }
    mbar_init(&ms->op_full, 256);
    mbar_init(&ms->a_full, 1);
    mbar_init(&ms->a_free, 128);
    mbar_init(&ms->am_full, 128);
    mbar_init(&ms->sst_full, 128);
    mbar_init(&ms->sst_free, 1);
    mbar_init(&ms->x_full, 1);
    mbar_init(&ms->x_free, 128);
    mbar_init(&ms->st_done, 1);
    mbar_init(&ms->fin, 1);
    mbar_init(&ms->w_done, 1);
    mbar_init(&ms->pobar, 256);
    mbar_init(&ms->nbar, 256);
    mbar_init(&ms->po_sync, 256);
    mbar_init(&ms->vst_empty, 256);
    // LayerNorm statistics: one arrival per epilogue warp of every other value slice
    for (int i = 0; i < 2; ++i) mbar_init(&ms->ln_full[i], 4 * (D / kDV - 1));
    ms->abort = 0;
    ms->never = 0;
    if (LN) fence_mbarrier_init_cluster();
  }
  if (LN && threadIdx.x < 64) {  // this slice's LayerNorm gain (1 when absent) and bias (0)
    const int h = bh % a.H, j = threadIdx.x & 31;
    const float* src = threadIdx.x < 32 ? a.ln_w : a.ln_b;
    reinterpret_cast<float*>(smem + CF::LNW_OFF)[threadIdx.x] =
        src ? src[(size_t)h * D + blockIdx.y * kDV + j] : (threadIdx.x < 32 ? 1.0f : 0.0f);
  }
  if (warp == 12) {
    tmem_alloc(&ms->tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (LN) cluster_sync_all();  // the other CTAs' barriers exist before any remote access

  if (warp < 8) {
    role_operands<D>(a, smem, ms, row0, nch);
  } else if (warp < 12) {
    role_epilogue<D, LN>(a, smem, ms, bh, row0, nch);
  } else if (warp == 12) {
    role_mma<D>(a, smem, ms, nch);
  } else if ((threadIdx.x & 31) == 0) {
    role_tma<D>(p, smem, ms, bh, nch);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    // every MMA has completed once `fin` fires (it is committed after the last one)
    if (!mbar_wait(&ms->fin, 0, &ms->never, 4000000000ull)) report(a.status, kErrTimeout);
    tc_fence_after();
    tmem_dealloc(ms->tmem, 512);
  }
  // LayerNorm: the other slices write statistics into this CTA's shared memory until their
  // last chunk; no CTA of the cluster exits before all have finished (every wait is bounded,
  // so every thread arrives here)
  if (LN) cluster_sync_all();
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

template <int D, bool LN>
cudaError_t launch_d(const FwdArgs& a, cudaStream_t stream) {
  // with the output LayerNorm the D / 32 value slices of a head form one cluster
  constexpr int kClY = LN ? D / kDV : 1;
  static std::atomic<uint64_t> attr_set{0};  // bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(chunk_kernel<D, LN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(BH, D / kDV, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg<D>::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = kClY;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kClY > 1 ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, chunk_kernel<D, LN>, p);
  count_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool chunk_supported(int d, int dtype, int causal) {
  return dtype == 0 && causal == 1 && (d == 64 || d == 128);
}

cudaError_t launch_fwd_chunk(const FwdArgs& a, cudaStream_t stream) {
  if (!a.scal) return cudaErrorInvalidValue;
  // at d = 64 only the fused-LayerNorm forward runs here (the plain one is the walk kernel's)
  if (a.d == 64) return a.ln ? launch_d<64, true>(a, stream) : cudaErrorInvalidValue;
  if (a.d == 128) return a.ln ? launch_d<128, true>(a, stream) : launch_d<128, false>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace zs
