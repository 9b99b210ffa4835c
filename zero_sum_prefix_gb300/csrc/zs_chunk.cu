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
//     W_{t,i} = a_t e_i + b_t s'_i + g_t k_i        (tensor core, hi/lo bf16 split, fp32 sum)
//     intra  S_{t,i} = [i <= t] (Q_t . K_i) W_{t,i} (fp32 product, rounded once to bf16)
//     Vsc_i = [ v_i | e_i v_i | s'_i v_i | k_i v_i ]                          (C x 128, bf16)
//     X[:, 0:96]   = Q [F~ | G | H]   (state of the previous chunks)
//     X[:, 96:128] = S V
//     o_t = a_t X_F + b_t X_G + g_t X_H + X_SV
//     state^T (128 x d; rows [unused | F~ | G | H]) += Vsc^T K, F~ rescaled by
//     e^{M_{c-1} - M_c} before each chunk's update.
//   The weight is formed to fp32 accuracy before the product is rounded: the three terms of w
//   nearly cancel (the weights sum to zero), so rounding them separately would amplify bf16
//   rounding errors.  The scalars s, m, Et = E e^{-m}, P follow the canonical blocked fp32 order
//   of zs_common.cuh (bit-identical to the decode step).
//
// Cluster pairs: the two CTAs of a cluster hold two value slices of the same (b, h).  Chunk c is
// owned by CTA c % 2: only the owner streams the chunk's q, k and u, computes its scalars
// (carries of the previous chunk arrive from the other CTA through distributed shared memory),
// rotates q and k and forms the weight operands and coefficients, then bulk-copies the rotated
// tiles, the weight operands and the coefficients into the other CTA's stage.  Each CTA builds
// its own scaled value tile, issues its own MMAs and writes its own output columns.  Stage
// releases and the weight-operand release are multicast to both CTAs.
//
// Warp roles (448 threads, one CTA per (b, h, value slice), one CTA per SM):
//   warps 0,1,4,5 (PS): warp w owns the 32-token block w of the chunk: the block's column sums,
//                     logits and local scalar chains (carries of earlier blocks through shared
//                     memory, two bounded barriers per chunk); hands (s, m, Et, P) per token and
//                     the chunk reference to PO through a ring (two slots, one with a cluster).
//   warps 2,3,6,7 (PO): per token row: rotary factors, rotate q/k in place (RoPE), norms, gates,
//                     row coefficients, the hi/lo weight operands and the scaled value tile Vsc.
//   warps 8-11  (E) : TMEM -> registers: S = masked (Q K^T) o W -> bf16 tile; state -> bf16
//                     tile (and the F~ rescale); X -> output rows.
//   warp 12     (M) : TMEM allocation; one elected thread issues every tcgen05.mma.
//   warp 13     (T) : TMA producers: lane 0 streams q and k chunks 128B-swizzled directly into
//                     the operand tiles (two stages at d = 64) and the value slice into a
//                     64B-swizzled staging tile, with an L2 prefetch of each chunk issued before
//                     its stage frees; lane 1 streams each chunk's u rows (one buffer).
// TMEM (512 columns): [0,128) Q K^T, [128,256) W, [256,384) X, [384, 384 + d) state^T.
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
constexpr int kCL = 1;  // CTAs per cluster (value slices sharing one (b, h)); 1 or 2
constexpr int kThreads = 448;
constexpr uint32_t kTile = 128 * 128;  // one [128 x 64] bf16 atom tile

__host__ __device__ constexpr uint32_t align_up(uint32_t x, uint32_t a) {
  return (x + a - 1) / a * a;
}

// Per-stage coefficients of a chunk: row coefficients (a, b, g), column scalars (e, s', k) and
// the chunk reference M_c; copied by the chunk's owner into the other CTA of the cluster.
struct Xch {
  float4 coef[kC];
  float cols[3][kC];
  float M;
  float pad[3];
};
static_assert(sizeof(Xch) == 3600, "Xch is moved by one bulk copy (multiple of 16 bytes)");

template <int D, int CL>
struct Cfg {
  static constexpr int KA = D / 64;               // atom tiles along d
  // Operand stages: NSV for the scaled value tile, NSQ for q, k and the Xch block.  With a
  // cluster at d = 64 the chunks of one owner are two apart; a third q/k stage lets an owner's
  // next chunk load while its previous chunk and the other CTA's chunk are in flight.
  static constexpr int NSV = (D == 64) ? 2 : 1;
  static constexpr int NSQ = (CL > 1 && D == 64) ? 3 : NSV;
  static constexpr int SCALS = (CL > 1) ? 1 : 2;  // slots of the scalar ring
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t K_OFF = Q_OFF + NSQ * KA * kTile;
  static constexpr uint32_t V_OFF = K_OFF + NSQ * KA * kTile;
  static constexpr uint32_t VST_OFF = V_OFF + NSV * 2 * kTile;   // raw v slice [128 x 32]
  static constexpr uint32_t SST_OFF = VST_OFF + 128 * 64;
  static constexpr uint32_t RW_OFF = SST_OFF + KA * kTile;       // weight MMA A: [128 x 16] bf16
  static constexpr uint32_t CW_OFF = RW_OFF + kC * 32;           // weight MMA B: [128 x 16] bf16
  static constexpr uint32_t XCH_OFF = CW_OFF + kC * 32;          // Xch [NSQ]
  static constexpr uint32_t U_OFF = align_up(XCH_OFF + NSQ * (uint32_t)sizeof(Xch), 1024);
  static constexpr uint32_t PHI_OFF = U_OFF + kC * D * 2;             // float [2][D/2] base angles
  static constexpr uint32_t THETA_OFF = PHI_OFF + 2 * (D / 2) * 4;    // float [D/2] frequencies
  static constexpr uint32_t LEND_OFF = THETA_OFF + (D / 2) * 4;       // float [4][D]
  static constexpr uint32_t BPUB_OFF = LEND_OFF + 4 * D * 4;         // float [4][4] + [2][4]
  static constexpr uint32_t CHAIN_OFF = BPUB_OFF + 128;               // float4 [4][32]
  static constexpr uint32_t SCAL_OFF = CHAIN_OFF + 4 * 32 * 16;     // float4 [SCALS][128]
  static constexpr uint32_t CIN_OFF = SCAL_OFF + SCALS * kC * 16;   // float [2][D] column carries
  static constexpr uint32_t KCIN_OFF = CIN_OFF + 2 * D * 4;         // float [2][4] scalar carries
  static constexpr uint32_t MISC_OFF = KCIN_OFF + 32;
  // output LayerNorm: per-row (mean, M2) of every value slice of the head, two chunk slots
  // (float2 [2][D / kDV][128]), then this slice's gain and bias (float [2][32]); only without
  // the chunk-alternating cluster, which has no room for them
  static constexpr uint32_t LNX_OFF = MISC_OFF + 512;
  static constexpr uint32_t LNW_OFF = LNX_OFF + (CL == 1 ? 2 * (D / kDV) * kC * 8 : 0);
  static constexpr uint32_t BYTES = LNW_OFF + (CL == 1 ? 2 * 32 * 4 : 0);
  static constexpr uint32_t SMEM = BYTES;  // the base is 1024-byte aligned (checked at entry)
  static constexpr uint32_t TM_A = 0, TM_W = 128, TM_X = 256, TM_ST = 384;
  // S tile (bf16 pairs, A operand of S V): its own 64 columns when d = 64, else the consumed
  // Q K^T columns (then the next Q K^T waits for the S V product)
  static constexpr uint32_t TM_S = (D == 64) ? 448 : 0;
  // bytes a non-owner receives per chunk: rotated Q and K, the weight operands, the Xch block
  static constexpr uint32_t PEER_BYTES = 2 * KA * kTile + 2 * kC * 32 + (uint32_t)sizeof(Xch);
  static_assert(SMEM <= 232448, "shared memory budget of one CTA");
};

struct Misc {
  uint64_t tma_full[2];
  uint64_t u_full, u_empty, vst_empty;
  uint64_t op_full, vsc_full;        // Vsc of an owned / other-owned chunk written
  uint64_t qk_empty[3];  // Q, K and Xch of a stage released by every CTA of the cluster
  uint64_t vsc_free[2];  // Vsc of the last chunk of this parity consumed (S V completed)
  uint64_t a_full, a_free, am_full, sst_full, sst_free, st_done, fin;
  uint64_t w_done;                   // both CTAs' weight MMAs have read R and C
  uint64_t x_full, x_free;
  uint64_t pbar;     // reusable barrier of the four scalar warps (bounded waits)
  uint64_t pobar;    // reusable barrier of the four operand warps
  uint64_t po_sync;  // Q, K, R, C and Xch of an owned chunk written
  uint64_t scal_full[2], scal_empty[2];
  uint64_t peer_full;            // tiles of a chunk owned by the other CTA have landed
  uint64_t ccar_full, kcar_full;  // carries from the other CTA's previous chunk
  uint64_t ln_full[2];  // output LayerNorm: row statistics of the other value slices landed
  float Mslot[2];
  int w_seen;  // with a cluster: number of w_done phases observed (monotonic)
  uint32_t tmem;
  int abort;
  int never;  // stays 0: lets the final waits ignore the abort flag
};

static_assert(sizeof(Misc) <= 512, "Misc fits its shared-memory slot");
static_assert(Cfg<64, 2>::NSQ <= 3 && Cfg<64, 1>::NSQ <= 3 && Cfg<128, 2>::NSQ <= 3,
              "qk_empty has one barrier per q/k stage");
static_assert(Cfg<64, 1>::SCALS <= 2 && Cfg<64, 2>::SCALS <= 2, "scal ring barriers");

struct ChunkParams {
  CUtensorMap tq, tk, tv;  // q, k: box {64, 128, 1} 128B swizzle; v: box {32, 128, 1} 64B swizzle
  CUtensorMap tu;          // u: box {d, 128, 1}, no swizzle (dense 2d-byte rows)
  FwdArgs a;
};

template <int CL>
__device__ __forceinline__ void fail_wait(Misc* ms, int* status) {
  report(status, kErrTimeout);
  ms->abort = 1;
  if (CL > 1) st_cluster_s32(mapa(smem_u32(&ms->abort), cluster_rank() ^ 1u), 1);
}

__device__ __forceinline__ Xch* xch(uint8_t* smem, uint32_t off, int st) {
  return reinterpret_cast<Xch*>(smem + off) + st;
}

// Load barrier of chunk c and the parity of its phase.  Without a cluster, one barrier per
// stage; with a cluster, one per owner, so that the operand warps (chunks of this CTA) and the
// epilogue warps (chunks of the other CTA) each wait for consecutive phases of their own barrier
// (a parity wait names its phase only when the previous phase has completed and the next one
// cannot have).
template <int D, int CL>
__device__ __forceinline__ int tf_index(int c) {
  return CL > 1 ? c % CL : c % Cfg<D, CL>::NSQ;
}
template <int D, int CL>
__device__ __forceinline__ uint32_t tf_phase(int c) {
  return (uint32_t)(CL > 1 ? c / CL : c / Cfg<D, CL>::NSQ) & 1u;
}

// Before the Vsc tile of chunk c is written: the S V product of chunk c - NS (same stage) has
// completed.  One barrier per chunk parity, so that each builder role (operand warps for this
// CTA's chunks, epilogue warps for the other CTA's) waits for consecutive phases of its own.
template <int D, int CL>
__device__ __forceinline__ bool vsc_wait(Misc* ms, int c) {
  constexpr int NS = Cfg<D, CL>::NSV;
  if (c < NS) return true;
  return mbar_wait_warp(&ms->vsc_free[(c - NS) & 1], (uint32_t)((c - NS) >> 1) & 1u, &ms->abort);
}

// Raw value row r (64B-swizzled staging tile) -> columns 0..31 of the Vsc tile (bf16 words).
__device__ __forceinline__ void copy_v_row(uint8_t* vt, const uint8_t* vst, int r) {
#pragma unroll
  for (int x = 0; x < 4; ++x)
    *reinterpret_cast<uint4*>(vt + sw128_off(r, x)) =
        *reinterpret_cast<const uint4*>(vst + sw64_off(r, x));
}

// Vsc row r: atom 0 = [v | e v], atom 1 = [s' v | k v] from the row's v (already in columns
// 0..31) and its column scalars (e, s', k).
__device__ __forceinline__ void build_vsc_row(uint8_t* vt, int r, float ce, float cs1, float ck) {
  const float2 ce2 = make_float2(ce, ce), cs2 = make_float2(cs1, cs1), ck2 = make_float2(ck, ck);
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const uint4 wv = *reinterpret_cast<const uint4*>(vt + sw128_off(r, x));
    const uint32_t pv[4] = {wv.x, wv.y, wv.z, wv.w};
    uint32_t pe[4], ps[4], pk[4];
#pragma unroll
    for (int y = 0; y < 4; ++y) {
      float2 v2;
      unpack_bf16x2(pv[y], v2.x, v2.y);
      const float2 e2 = __fmul2_rn(ce2, v2), s2 = __fmul2_rn(cs2, v2), k2 = __fmul2_rn(ck2, v2);
      pe[y] = pack_bf16x2(e2.x, e2.y);
      ps[y] = pack_bf16x2(s2.x, s2.y);
      pk[y] = pack_bf16x2(k2.x, k2.y);
    }
    *reinterpret_cast<uint4*>(vt + sw128_off(r, 4 + x)) = make_uint4(pe[0], pe[1], pe[2], pe[3]);
    *reinterpret_cast<uint4*>(vt + kTile + sw128_off(r, x)) = make_uint4(ps[0], ps[1], ps[2], ps[3]);
    *reinterpret_cast<uint4*>(vt + kTile + sw128_off(r, 4 + x)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
}

// Warps 0, 1, 4, 5 are the scalar warps and 2, 3, 6, 7 the operand warps (warp w runs on
// sub-partition w % 4, so each of these sub-partitions interleaves one role's code with the
// epilogue's); both roles number their warps 0..3 in this order.
__device__ __forceinline__ int group_index() {
  const int warp = threadIdx.x >> 5;
  return (warp & 1) | ((warp >> 2) << 1);
}

// ============================================================================ T: TMA producer
// Every CTA streams its value slice for every chunk; q and k only for the chunks it owns.
template <int D, int CL>
__device__ void role_tma(const ChunkParams& p, uint8_t* smem, Misc* ms, int bh, int nch,
                         int rank) {
  using CF = Cfg<D, CL>;
  const uint32_t base = smem_u32(smem);
  const int j0 = blockIdx.y * kDV;
  constexpr uint32_t qk_bytes = 2 * CF::KA * kTile, v_bytes = 128 * 64;
  tma_prefetch_desc(&p.tq);
  tma_prefetch_desc(&p.tk);
  tma_prefetch_desc(&p.tv);
  for (int c = 0; c < nch; ++c) {
    const int st = c % CF::NSQ;
    const bool owned = (c % CL) == rank;
    if (c >= CF::NSQ) {
      // the chunk's tiles start towards L2 while the stage is still in use
      if (owned) {
#pragma unroll
        for (int at = 0; at < CF::KA; ++at) {
          tma_prefetch_3d(&p.tq, 64 * at, c * kC, bh);
          tma_prefetch_3d(&p.tk, 64 * at, c * kC, bh);
        }
      }
      tma_prefetch_3d(&p.tv, j0, c * kC, bh);
      // both CTAs of the cluster have released the stage's Q, K and Xch
      if (!mbar_wait_cl(&ms->qk_empty[st], ((c / CF::NSQ) - 1) & 1, &ms->abort)) {
        fail_wait<CL>(ms, p.a.status);
        return;
      }
    }
    // a chunk owned by the other CTA: its tiles arrive by bulk copy; the barrier's previous
    // phase (the other CTA's previous chunk) must have completed before this arrival
    if (CL > 1 && !owned) {
      if (c >= CL && !mbar_wait_cl(&ms->peer_full, (uint32_t)((c - CL) / CL) & 1u, &ms->abort)) {
        fail_wait<CL>(ms, p.a.status);
        return;
      }
      mbar_arrive_expect_tx(&ms->peer_full, CF::PEER_BYTES);
    }
    uint64_t* tf = &ms->tma_full[tf_index<D, CL>(c)];
    mbar_arrive_expect_tx(tf, (owned ? qk_bytes : 0u) + v_bytes);
    if (owned) {
      const uint32_t qt = base + CF::Q_OFF + st * CF::KA * kTile;
      const uint32_t kt = base + CF::K_OFF + st * CF::KA * kTile;
#pragma unroll
      for (int at = 0; at < CF::KA; ++at) {
        tma_load_3d(qt + at * kTile, &p.tq, 64 * at, c * kC, bh, tf);
        tma_load_3d(kt + at * kTile, &p.tk, 64 * at, c * kC, bh, tf);
      }
    }
    // the raw value slice has one buffer, released by the operand warps once copied
    if (c >= 1 && !mbar_wait(&ms->vst_empty, (c - 1) & 1, &ms->abort)) {
      fail_wait<CL>(ms, p.a.status);
      return;
    }
    tma_load_3d(base + CF::VST_OFF, &p.tv, j0, c * kC, bh, tf);
  }
}

// With a cluster: observes every phase of w_done in order and publishes the count, for the
// operand warps, which only handle every other chunk (a parity wait names its phase only when
// the waiter has seen the previous one).
template <int CL>
__device__ void role_wdone_observer(const FwdArgs& a, Misc* ms, int nch) {
  for (int c = 0; c < nch; ++c) {
    if (!mbar_wait_cl(&ms->w_done, (uint32_t)c & 1u, &ms->abort)) {
      fail_wait<CL>(ms, a.status);
      return;
    }
    st_release_s32(&ms->w_seen, c + 1);
  }
}

// u rows of each owned chunk (single buffer, released by the scalar warps after their logits);
// a separate producer thread so that this stream never waits behind the operand stages.
template <int D, int CL>
__device__ void role_tma_u(const ChunkParams& p, uint8_t* smem, Misc* ms, int bh, int nch,
                           int rank) {
  using CF = Cfg<D, CL>;
  const uint32_t base = smem_u32(smem);
  tma_prefetch_desc(&p.tu);
  for (int c = rank, kk = 0; c < nch; c += CL, ++kk) {
    if (kk >= 1) {
      tma_prefetch_3d(&p.tu, 0, c * kC, bh);
      if (!mbar_wait(&ms->u_empty, (kk - 1) & 1, &ms->abort)) {
        fail_wait<CL>(ms, p.a.status);
        return;
      }
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
// Runs the chunks this CTA owns.  With a cluster, the column carry at a chunk's start and the
// chunk-start scalar carries (mC, EC, CP) come from the other CTA, which processed the previous
// chunk; the carries of the next chunk are sent the same way.  Slots are indexed by the number
// of carries received so far: a slot is rewritten only two owned chunks later.
template <int D, int CL>
__device__ void role_scalars(const FwdArgs& a, uint8_t* smem, Misc* ms, int bh, int h,
                             size_t row0, int nch, int rank) {
  using CF = Cfg<D, CL>;
  constexpr int R = D / 32;
  constexpr int RP = (R + 1) / 2;  // column pairs per lane (R = 1 uses the .x half only)
  const int w = group_index(), lane = threadIdx.x & 31;  // w: the warp's 32-token block
  const int r = 32 * w + lane;     // token row inside the chunk, 0..127
  const int N = a.N;
  float* lend = reinterpret_cast<float*>(smem + CF::LEND_OFF);      // [4][D]
  float* bpub = reinterpret_cast<float*>(smem + CF::BPUB_OFF);      // [4][4] + kc [2][4]
  float4* chain = reinterpret_cast<float4*>(smem + CF::CHAIN_OFF);  // [4][32] (s, f, g, -)
  float4* scal = reinterpret_cast<float4*>(smem + CF::SCAL_OFF);    // [2][128] (s, m, Et, P)
  const float* cin = reinterpret_cast<const float*>(smem + CF::CIN_OFF);    // [2][D]
  const float* kcin = reinterpret_cast<const float*>(smem + CF::KCIN_OFF);  // [2][4]
  const uint32_t peer = (uint32_t)rank ^ 1u;
  const bool dbg = blockIdx.y < CL;  // the first cluster of value slices writes the scalars
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
  if (CL == 1 && r == 0) {
    bpub[16 + 0] = -INFINITY;  // chunk-start carries (mC, EC, CP) for chunk 0
    bpub[16 + 1] = 0.0f;
    bpub[16 + 2] = 0.0f;
  }

  for (int c = rank, kk = 0; c < nch; c += CL, ++kk) {
    const int slot = kk % CF::SCALS;
    const int i = c * kC + r;
    const bool valid = i < N;
    const int b0 = c * kC + 32 * w;  // first token of this warp's block
    const int nvalid = max(0, min(32, N - b0));
    const int rslot = ((c - 1) / 2) & 1;  // carry slot of this chunk (cluster of two)
    // ---- u of the block from the staged tile: lane owns columns R lane .. R lane + R - 1 ----
    if (!mbar_wait_warp(&ms->u_full, kk & 1, &ms->abort)) {
      fail_wait<CL>(ms, a.status);
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
    if (!mbar_wait_warp(&ms->pbar, (2 * kk) & 1, &ms->abort)) {
      fail_wait<CL>(ms, a.status);
      return;
    }
    // ---- column carry at this block's start (and at the next chunk's start) ----
    if (CL > 1 && c > 0) {
      if (!mbar_wait_cl_warp(&ms->ccar_full, rslot, &ms->abort)) {
        fail_wait<CL>(ms, a.status);
        return;
      }
#pragma unroll
      for (int x = 0; x < RP; ++x)
        Cc[x] = make_float2(cin[rslot * D + R * lane + 2 * x],
                            R > 1 ? cin[rslot * D + R * lane + 2 * x + 1] : 0.0f);
    }
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
    if (CL > 1 && w == 0 && c + 1 < nch) {  // the next chunk's column carry -> other CTA
      const uint32_t dst = mapa(smem_u32(smem + CF::CIN_OFF) + (uint32_t)(((c / 2) & 1) * D * 4),
                                peer);
#pragma unroll
      for (int x = 0; x < RP; ++x) {
        st_cluster_f32(dst + (uint32_t)(R * lane + 2 * x) * 4, Cc[x].x);
        if (R > 1) st_cluster_f32(dst + (uint32_t)(R * lane + 2 * x + 1) * 4, Cc[x].y);
      }
      mbar_arrive_remote(mapa(smem_u32(&ms->ccar_full), peer));
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
    if (!mbar_wait_warp(&ms->pbar, (2 * kk + 1) & 1, &ms->abort)) {
      fail_wait<CL>(ms, a.status);
      return;
    }
    // carries at this block's start: chunk-start carries folded over the earlier blocks
    BlockCarry kw{-INFINITY, 0.0f, 0.0f};
    if (CL == 1) {
      const float* kcb = bpub + 16 + (c & 1) * 4;
      kw = BlockCarry{kcb[0], kcb[1], kcb[2]};
    } else if (c > 0) {
      if (!mbar_wait_cl_warp(&ms->kcar_full, rslot, &ms->abort)) {
        fail_wait<CL>(ms, a.status);
        return;
      }
      kw = BlockCarry{kcin[rslot * 4 + 0], kcin[rslot * 4 + 1], kcin[rslot * 4 + 2]};
    }
    for (int ww = 0; ww < w; ++ww) fold_block(kw, bpub[ww * 4 + 0], bpub[ww * 4 + 1], bpub[ww * 4 + 2]);
    float M = kw.mC;  // running max at the chunk's last valid token (max is exact)
#pragma unroll
    for (int ww = 0; ww < 4; ++ww) M = fmaxf(M, bpub[ww * 4 + 1]);
    if (w == 3 && lane == 0) {  // chunk-start carries of the next chunk
      BlockCarry kn = kw;
      fold_block(kn, bpub[12 + 0], bpub[12 + 1], bpub[12 + 2]);
      if (CL == 1) {
        float* kcn = bpub + 16 + ((c + 1) & 1) * 4;
        kcn[0] = kn.mC;
        kcn[1] = kn.EC;
        kcn[2] = kn.CP;
      } else if (c + 1 < nch) {
        const uint32_t dst =
            mapa(smem_u32(smem + CF::KCIN_OFF) + (uint32_t)(((c / 2) & 1) * 16), peer);
        st_cluster_f32(dst + 0, kn.mC);
        st_cluster_f32(dst + 4, kn.EC);
        st_cluster_f32(dst + 8, kn.CP);
        mbar_arrive_remote(mapa(smem_u32(&ms->kcar_full), peer));
      }
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
    // hand the scalars to the operand warps (ring of SCALS slots)
    if (kk >= CF::SCALS &&
        !mbar_wait_warp(&ms->scal_empty[slot], ((kk / CF::SCALS) - 1) & 1, &ms->abort)) {
      fail_wait<CL>(ms, a.status);
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
// Chunks this CTA owns: rotate q/k, coefficients, weight operands and the Xch block (bulk-copied
// to the other CTA of the cluster), then this CTA's scaled value tile Vsc.  The value tiles of
// the chunks of the other CTA are built by the epilogue warps.
template <int D, int CL>
__device__ void role_operands(const FwdArgs& a, uint8_t* smem, Misc* ms, int h, size_t row0,
                              int nch, int rank) {
  using CF = Cfg<D, CL>;
  const int w = group_index(), lane = threadIdx.x & 31;  // w: the warp's 32-row group
  const int r = 32 * w + lane;      // token row inside the chunk, 0..127
  const int N = a.N;
  const float4* scal = reinterpret_cast<const float4*>(smem + CF::SCAL_OFF);
  float* phi = reinterpret_cast<float*>(smem + CF::PHI_OFF);      // [2][D/2]
  float* theta = reinterpret_cast<float*>(smem + CF::THETA_OFF);  // [D/2]
  const uint32_t peer = (uint32_t)rank ^ 1u;
  const double two_pi = 6.283185307179586476925286766559;
  constexpr int PPW = (D / 2 + 3) / 4;  // rotary pairs per warp
  const int pj = w * PPW + lane;
  const bool owns_pair = a.rope && lane < PPW && pj < D / 2;
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
  // gate logits of chunk cc (loaded one chunk ahead so that their latency is hidden); x0 is the
  // optional zero-order gate (-inf when absent, so that its sigmoid is 0)
  auto load_gates = [&](int cc, float& x1, float& xh, float& x0) {
    x1 = 0.0f;
    xh = 0.0f;
    x0 = -INFINITY;
    if (cc < nch && cc * kC + r < N) {
      x1 = __ldg(a.g1 + row0 + cc * kC + r);
      xh = __ldg(a.gh + row0 + cc * kC + r);
      if (a.g0) x0 = __ldg(a.g0 + row0 + cc * kC + r);
    }
  };
  float g1, gh, g0;
  load_gates(rank, g1, gh, g0);
  put_phi(rank, 0);

  for (int c = rank, kk = 0; c < nch; c += CL, ++kk) {
    const int st = c % CF::NSQ;
    const int i = c * kC + r;
    const bool valid = i < N;
    Xch* xc = xch(smem, CF::XCH_OFF, st);
    mbar_arrive(&ms->pobar);
    if (!mbar_wait_warp(&ms->pobar, kk & 1, &ms->abort)) {
      fail_wait<CL>(ms, a.status);
      return;
    }
    if (!mbar_wait_warp(&ms->tma_full[tf_index<D, CL>(c)], tf_phase<D, CL>(c), &ms->abort)) {
      fail_wait<CL>(ms, a.status);
      return;
    }
    uint8_t* qt = smem + CF::Q_OFF + st * CF::KA * kTile;
    uint8_t* kt = smem + CF::K_OFF + st * CF::KA * kTile;
    uint8_t* vt = smem + CF::V_OFF + (c % CF::NSV) * 2 * kTile;
    float g1n, ghn, g0n;
    load_gates(c + CL, g1n, ghn, g0n);
    float ce = 0.0f, cs1 = 0.0f, ck = 0.0f;
    {
      // ---- rotate q, k in place (TMA tiles), norms ----
      const bool rot = a.rope != 0 && valid;
      float2 qq2 = make_float2(0.0f, 0.0f), kk2 = make_float2(0.0f, 0.0f);
      const float* ph = phi + (kk & 1) * (D / 2);
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
      const float qq = __fadd_rn(qq2.x, qq2.y), kq = __fadd_rn(kk2.x, kk2.y);
      // ---- scalars of this token from the scalar warps ----
      const int slot = kk % CF::SCALS;
      if (!mbar_wait_warp(&ms->scal_full[slot], (kk / CF::SCALS) & 1, &ms->abort)) {
        fail_wait<CL>(ms, a.status);
        return;
      }
      const float4 sc = scal[slot * kC + r];
      const float M = ms->Mslot[slot];
      mbar_arrive(&ms->scal_empty[slot]);
      const float s = sc.x, m = sc.y, Et = sc.z, P = sc.w;
      // column scalars and row coefficients (these feed bf16 / fp32 products, not the scalar
      // contract: fast exp, reciprocal square root and division are accurate enough here)
      const float kap = rsqrtf(fmaxf(kq, 1e-24f));
      const float rho = rsqrtf(fmaxf(qq, 1e-24f));
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
        if (a.g0) cf.z += rho * __fdividef(1.0f, 1.0f + __expf(-g0)) * rt;  // zero-order term
        if (!isfinite(cf.x) || !isfinite(ce)) report(a.status, kErrRange);
      }
      xc->coef[r] = cf;
      xc->cols[0][r] = ce;
      xc->cols[1][r] = cs1;
      xc->cols[2][r] = ck;
      if (r == 0) xc->M = M;
      // Weight operands: W_{t,i} = a_t e_i + b_t s'_i + g_t k_i is formed by one K = 16 MMA of
      // the row vector [a a' a a' b b' b b' g g' g g' 0 0 0 0] (hi and lo bf16 parts,
      // x = x + x') and the column vector [e e' e e' s s' s s' k k' k k' 0 0 0 0] paired as
      // (hi hi, hi lo, lo hi, lo lo): every product is exact in fp32, the representation error
      // is about 2^-17 of each term, so the nearly cancelling sum keeps fp32-level accuracy.
      // The buffer is single: both CTAs' weight MMAs of the previous chunk must have completed
      // (without a cluster these warps wait for every phase of w_done in order; with one, the
      // observer thread's count says how many phases completed).
      bool wok = true;
      if (c >= 1) {
        wok = CL > 1 ? counter_wait(&ms->w_seen, c, &ms->abort)
                     : mbar_wait(&ms->w_done, (c - 1) & 1, &ms->abort);
      }
      if (!__all_sync(0xffffffffu, wok)) {
        fail_wait<CL>(ms, a.status);
        return;
      }
      {
        float xh[6], xl[6];
        const float xs[6] = {cf.x, cf.y, cf.z, ce, cs1, ck};
#pragma unroll
        for (int k = 0; k < 6; ++k) {
          xh[k] = __bfloat162float(__float2bfloat16_rn(xs[k]));
          xl[k] = __fsub_rn(xs[k], xh[k]);
        }
        uint8_t* rw = smem + CF::RW_OFF;
        uint8_t* cw = smem + CF::CW_OFF;
        *reinterpret_cast<uint4*>(rw + sw32_off(r, 0)) =
            make_uint4(pack_bf16x2(xh[0], xh[0]), pack_bf16x2(xl[0], xl[0]),
                       pack_bf16x2(xh[1], xh[1]), pack_bf16x2(xl[1], xl[1]));
        *reinterpret_cast<uint4*>(rw + sw32_off(r, 1)) =
            make_uint4(pack_bf16x2(xh[2], xh[2]), pack_bf16x2(xl[2], xl[2]), 0u, 0u);
        *reinterpret_cast<uint4*>(cw + sw32_off(r, 0)) =
            make_uint4(pack_bf16x2(xh[3], xl[3]), pack_bf16x2(xh[3], xl[3]),
                       pack_bf16x2(xh[4], xl[4]), pack_bf16x2(xh[4], xl[4]));
        *reinterpret_cast<uint4*>(cw + sw32_off(r, 1)) =
            make_uint4(pack_bf16x2(xh[5], xl[5]), pack_bf16x2(xh[5], xl[5]), 0u, 0u);
      }
      // Q, K, R, C and Xch are complete: the MMA may start, and with a cluster one thread
      // bulk-copies them to the other CTA once every operand thread's writes are visible to the
      // copy engine
      fence_proxy_async_smem();
      mbar_arrive(&ms->po_sync);
      if (CL > 1 && r == 0) {
        if (!mbar_wait(&ms->po_sync, kk & 1, &ms->abort)) {
          fail_wait<CL>(ms, a.status);
          return;
        }
        const uint32_t bar = mapa(smem_u32(&ms->peer_full), peer);
        const uint32_t lq = smem_u32(qt), lk = smem_u32(kt);
        const uint32_t lw = smem_u32(smem + CF::RW_OFF), lx = smem_u32(xc);
        bulk_copy_to_cta(mapa(lq, peer), lq, CF::KA * kTile, bar);
        bulk_copy_to_cta(mapa(lk, peer), lk, CF::KA * kTile, bar);
        bulk_copy_to_cta(mapa(lw, peer), lw, 2 * kC * 32, bar);
        bulk_copy_to_cta(mapa(lx, peer), lx, (uint32_t)sizeof(Xch), bar);
      }
    }
    // value slice of this token: raw bf16 words copied to columns 0..31 of the Vsc tile (once the
    // stage's previous Vsc was consumed), the staging buffer handed back, then the scaled parts
    if (!vsc_wait<D, CL>(ms, c)) {
      fail_wait<CL>(ms, a.status);
      return;
    }
    copy_v_row(vt, smem + CF::VST_OFF, r);
    mbar_arrive(&ms->vst_empty);
    build_vsc_row(vt, r, ce, cs1, ck);
    fence_proxy_async_smem();
    mbar_arrive(&ms->op_full);
    if (c + CL < nch) put_phi(c + CL, (kk + 1) & 1);
    g1 = g1n;
    gh = ghn;
    g0 = g0n;
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
// qk_empty follows the Q [F|G|H] product (the S V product for the first chunk).  w_done and
// qk_empty are delivered to both CTAs of a cluster (the owner of a later chunk writes into the
// other CTA's buffers).  The epilogue reads a chunk's Xch block before it frees X of the
// previous chunk, which the Q [F|G|H] product waits for.
template <int D, int CL>
__device__ void role_mma(const FwdArgs& a, uint8_t* smem, Misc* ms, int nch) {
  constexpr uint16_t kAll = (uint16_t)((1u << CL) - 1u);  // every CTA of the cluster
  using CF = Cfg<D, CL>;
  const uint32_t base = smem_u32(smem);
  const uint32_t tm = ms->tmem;
  const uint32_t tA = tm + CF::TM_A, tW = tm + CF::TM_W, tX = tm + CF::TM_X, tS = tm + CF::TM_ST;
  constexpr uint32_t id_qk = idesc_bf16_f32(128, 128, false, false);   // Q K^T, R C^T
  constexpr uint32_t id_qs = idesc_bf16_f32(128, 96, false, false);    // Q [F|G|H]
  constexpr uint32_t id_sv = idesc_bf16_f32(128, 32, false, true);     // S V
  constexpr uint32_t id_st = idesc_bf16_f32(128, D, true, true);       // Vsc^T K
  const uint64_t d_rw = sw32_desc(base + CF::RW_OFF), d_cw = sw32_desc(base + CF::CW_OFF);
  bool ok = true;
  const int rank = CL > 1 ? (int)cluster_rank() : 0;
  for (int c = 0; c < nch && ok; ++c) {
    const int st = c % CF::NSQ;
    const bool owned = (c % CL) == rank;
    const uint32_t ph = (uint32_t)(c / CL) & 1u;  // phase of the owned / other-owned barriers
    const uint32_t qt = base + CF::Q_OFF + st * CF::KA * kTile;
    const uint32_t kt = base + CF::K_OFF + st * CF::KA * kTile;
    const uint32_t vt = base + CF::V_OFF + (c % CF::NSV) * 2 * kTile;
    ok = owned ? mbar_wait(&ms->po_sync, ph, &ms->abort)
               : mbar_wait_cl(&ms->peer_full, ph, &ms->abort);
    if (ok && c >= 1) ok = mbar_wait(&ms->a_free, (c - 1) & 1, &ms->abort);
    // the S tile shares the Q K^T columns: the previous S V product must have read it
    if (CF::TM_S == CF::TM_A && ok && c >= 1) ok = mbar_wait(&ms->x_full, (c - 1) & 1, &ms->abort);
    // every phase of w_done is observed in order (the end-of-kernel wait relies on it)
    if (ok && c >= 1) ok = mbar_wait_cl(&ms->w_done, (c - 1) & 1, &ms->abort);
    if (!ok) break;
    tc_fence_after();
    // ---- A = Q K^T (K = d); W = R C^T (K = 16) ----
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk / 4) * kTile + (kk % 4) * 32;
      mma_bf16(tA, sw128_desc(qt + off, 16, 1024), sw128_desc(kt + off, 16, 1024), id_qk,
               kk > 0);
    }
    mma_bf16(tW, d_rw, d_cw, id_qk, 0u);
    mma_commit(&ms->a_full);
    if (CL > 1) mma_commit_mc(&ms->w_done, kAll);
    else mma_commit(&ms->w_done);
    // ---- state^T += Vsc^T K (M = 128 value rows, N = d, K = chunk tokens) ----
    if (c >= 1 && !mbar_wait(&ms->sst_full, (c - 1) & 1, &ms->abort)) { ok = false; break; }
    ok = owned ? mbar_wait(&ms->op_full, ph, &ms->abort) : mbar_wait(&ms->vsc_full, ph, &ms->abort);
    if (!ok) break;
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < kC / 16; ++kk) {
      const uint32_t off = kk * 2048;
      mma_bf16(tS, sw128_desc(vt + off, kTile, 1024), sw128_desc(kt + off, kTile, 1024), id_st,
               (c > 0 || kk > 0) ? 1u : 0u);
    }
    mma_commit(&ms->st_done);
    // ---- X[:, 0:96] = Q [F~ | G | H] (state of the previous chunks, B tile rows 32..127) ----
    if (c >= 1) {
      if (!mbar_wait(&ms->x_free, (c - 1) & 1, &ms->abort)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sst = base + CF::SST_OFF + 32 * 128;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk / 4) * kTile + (kk % 4) * 32;
        mma_bf16(tX, sw128_desc(qt + off, 16, 1024), sw128_desc(sst + off, 16, 1024), id_qs,
                 kk > 0);
      }
      mma_commit(&ms->sst_free);
      // Q, K (and, through the epilogue's order, Xch) of this chunk are no longer read
      if (CL > 1) mma_commit_mc(&ms->qk_empty[st], kAll);
      else mma_commit(&ms->qk_empty[st]);
    }
    // ---- X[:, 96:128] = S V ----
    if (!mbar_wait(&ms->am_full, c & 1, &ms->abort)) { ok = false; break; }
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < kC / 16; ++kk) {
      const uint32_t boff = kk * 2048;  // MN-major B, 16 token rows per step
      mma_bf16_ts(tX + 96, tm + CF::TM_S + kk * 8, sw128_desc(vt + boff, kTile, 1024), id_sv,
                  kk > 0);
    }
    mma_commit(&ms->x_full);
    if (c == 0) {  // the first chunk has no Q [F|G|H] product: release after the S tile was read
      if (CL > 1) mma_commit_mc(&ms->qk_empty[st], kAll);
      else mma_commit(&ms->qk_empty[st]);
    }
    mma_commit(&ms->vsc_free[c & 1]);
  }
  if (!ok) fail_wait<CL>(ms, a.status);
  mma_commit(&ms->fin);
}

// ============================================================================ E: epilogue
// Per chunk c: the S tile (A o W, masked, bf16), the scaled value tile of chunk c+1 when the
// other CTA of the cluster owns it, the state after chunk c as the bf16 B tile of chunk c+1 (F~
// rescaled to M_{c+1}), then the output rows of chunk c.
template <int D, int CL, bool LN>
__device__ void role_epilogue(const FwdArgs& a, uint8_t* smem, Misc* ms, int bh, size_t row0,
                              int nch) {
  using CF = Cfg<D, CL>;
  const int wq = (threadIdx.x >> 5) & 3;          // TMEM lane quadrant of this warp
  const int t = wq * 32 + (threadIdx.x & 31);     // TMEM lane = token row / state row
  const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
  const uint32_t tm = ms->tmem + lane_off;
  const uint32_t base = smem_u32(smem);
  const int j0 = blockIdx.y * kDV;
  const int N = a.N;
  __nv_bfloat16* __restrict__ out = static_cast<__nv_bfloat16*>(a.out) + row0 * D;
  const int rank = CL > 1 ? (int)cluster_rank() : 0;
  auto owned = [&](int cc) { return (cc % CL) == rank; };
  // coefficients and M of chunk cc are in this CTA's Xch block
  auto wait_xch = [&](int cc) -> bool {
    const uint32_t ph = (uint32_t)(cc / CL) & 1u;
    return owned(cc) ? mbar_wait_warp(&ms->po_sync, ph, &ms->abort)
                     : mbar_wait_cl_warp(&ms->peer_full, ph, &ms->abort);
  };
  // value tile of a chunk owned by the other CTA (row t)
  auto vsc_other = [&](int cc) -> bool {
    const int sv = cc % CF::NSV;
    if (!mbar_wait_warp(&ms->tma_full[tf_index<D, CL>(cc)], tf_phase<D, CL>(cc), &ms->abort))
      return false;
    if (!vsc_wait<D, CL>(ms, cc)) return false;
    uint8_t* vt = smem + CF::V_OFF + sv * 2 * kTile;
    copy_v_row(vt, smem + CF::VST_OFF, t);
    mbar_arrive(&ms->vst_empty);
    if (!mbar_wait_cl_warp(&ms->peer_full, (uint32_t)(cc / CL) & 1u, &ms->abort)) return false;
    const Xch* xv = xch(smem, CF::XCH_OFF, cc % CF::NSQ);
    build_vsc_row(vt, t, xv->cols[0][t], xv->cols[1][t], xv->cols[2][t]);
    fence_proxy_async_smem();
    mbar_arrive(&ms->vsc_full);
    return true;
  };
  bool ok = true;
  if (CL > 1 && nch > 0 && !owned(0)) ok = vsc_other(0);
  // (a, b, g) of row t and M of the current chunk: read while the previous chunk is in flight
  // (before X of that chunk is freed), since the chunk's Xch block is released with its Q, K
  float4 cf = make_float4(0.f, 0.f, 0.f, 0.f);
  float M_cur = 0.0f;
  if (ok && nch > 0) {
    ok = wait_xch(0);
    cf = xch(smem, CF::XCH_OFF, 0)->coef[t];
    M_cur = xch(smem, CF::XCH_OFF, 0)->M;
  }
  for (int c = 0; c < nch && ok; ++c) {
    float4 cf_next = make_float4(0.f, 0.f, 0.f, 0.f);
    float M_next = 0.0f;
    // ---- S = [i <= t] (Q K^T) o W, fp32 product then bf16 (rows t, K = token i) ----
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
          const int col = 16 * h + 2 * y;
          if ((h >> 1) == wq) {  // diagonal block: keep i <= t only
            if (col > t) val.x = 0.0f;
            if (col + 1 > t) val.y = 0.0f;
          }
          pw[y] = pack_bf16x2(val.x, val.y);
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
    if (CL > 1 && c + 1 < nch && !owned(c + 1)) {
      ok = vsc_other(c + 1);
      if (!ok) break;
    }
    // ---- state after chunk c -> bf16 B operand rows 32..127 of chunk c+1, F~ rescaled ----
    if (c + 1 < nch) {
      const int st1 = (c + 1) % CF::NSQ;
      ok = wait_xch(c + 1);
      if (ok) ok = mbar_wait_warp(&ms->st_done, c & 1, &ms->abort);
      if (ok && c >= 1) ok = mbar_wait_warp(&ms->sst_free, (c - 1) & 1, &ms->abort);
      if (!ok) break;
      const Xch* xn = xch(smem, CF::XCH_OFF, st1);
      cf_next = xn->coef[t];
      M_next = xn->M;
      tc_fence_after();
      if (wq >= 1) {
        const bool rescale = (wq == 1) && (M_next > M_cur);
        const float fac = rescale ? expf(__fsub_rn(M_cur, M_next)) : 1.0f;
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
#pragma unroll
          for (int q = 0; q < 2; ++q) {
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              const uint32_t* w8 = rr[q] + 8 * x;
              uint4 p;
              p.x = pack_bf16x2(__uint_as_float(w8[0]), __uint_as_float(w8[1]));
              p.y = pack_bf16x2(__uint_as_float(w8[2]), __uint_as_float(w8[3]));
              p.z = pack_bf16x2(__uint_as_float(w8[4]), __uint_as_float(w8[5]));
              p.w = pack_bf16x2(__uint_as_float(w8[6]), __uint_as_float(w8[7]));
              const int col0 = c0 + 16 * q + 8 * x;
              sts128(sst + (col0 / 64) * kTile + sw128_off(t, (col0 % 64) / 8), p);
            }
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
        tc_fence_before();
        mbar_arrive(&ms->x_free);
      }
      if (i < N) {
        dst[2 * hf + 0] = make_uint4(ob[0], ob[1], ob[2], ob[3]);
        dst[2 * hf + 1] = make_uint4(ob[4], ob[5], ob[6], ob[7]);
      }
    }
    cf = cf_next;
    M_cur = M_next;
  }
  if (!ok) {
    fail_wait<CL>(ms, a.status);
    return;
  }
  // ---- final state (prefill): columns j0.. of F~, G, H (state rows 32..127) ----
  if (a.final_state && nch > 0) {
    if (!mbar_wait_warp(&ms->st_done, (nch - 1) & 1, &ms->abort)) {
      fail_wait<CL>(ms, a.status);
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
template <int D, int CL, bool LN>
__global__ void __launch_bounds__(kThreads, 1) chunk_kernel(const __grid_constant__ ChunkParams p) {
  using CF = Cfg<D, CL>;
  const FwdArgs& a = p.a;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (smem_u32(smem) & 1023u) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) report(a.status, kErrUnsupported);
    return;
  }
  Misc* ms = reinterpret_cast<Misc*>(smem + CF::MISC_OFF);
  const int warp = threadIdx.x >> 5;
  const int bh = blockIdx.x, h = bh % a.H;
  const size_t row0 = (size_t)bh * a.N;
  const int nch = (a.N + kC - 1) / kC;
  const int rank = CL > 1 ? (int)cluster_rank() : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms->tma_full[i], 1);
      mbar_init(&ms->vsc_free[i], 1);
    }
    for (int i = 0; i < 3; ++i) mbar_init(&ms->qk_empty[i], CL);
    mbar_init(&ms->op_full, 128);
    mbar_init(&ms->vsc_full, 128);
    mbar_init(&ms->a_full, 1);
    mbar_init(&ms->a_free, 128);
    mbar_init(&ms->am_full, 128);
    mbar_init(&ms->sst_full, 128);
    mbar_init(&ms->sst_free, 1);
    mbar_init(&ms->x_full, 1);
    mbar_init(&ms->x_free, 128);
    mbar_init(&ms->st_done, 1);
    mbar_init(&ms->fin, 1);
    mbar_init(&ms->w_done, CL);
    mbar_init(&ms->pbar, 128);
    mbar_init(&ms->pobar, 128);
    mbar_init(&ms->po_sync, 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms->scal_full[i], 128);
      mbar_init(&ms->scal_empty[i], 128);
    }
    mbar_init(&ms->u_full, 1);
    mbar_init(&ms->u_empty, 128);
    mbar_init(&ms->vst_empty, 128);
    mbar_init(&ms->peer_full, 1);
    mbar_init(&ms->ccar_full, 32);
    mbar_init(&ms->kcar_full, 1);
    // LayerNorm statistics: one arrival per epilogue warp of every other value slice
    for (int i = 0; i < 2; ++i) mbar_init(&ms->ln_full[i], 4 * (D / kDV - 1));
    ms->abort = 0;
    ms->never = 0;
    ms->w_seen = 0;
    if (CL > 1 || LN) fence_mbarrier_init_cluster();
  }
  if (LN && threadIdx.x < 64) {  // this slice's LayerNorm gain (1 when absent) and bias (0)
    const int j = threadIdx.x & 31;
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
  if (CL > 1 || LN) cluster_sync_all();  // the other CTAs' barriers exist before any remote access

  if (warp < 8 && (warp & 2) == 0) {
    role_scalars<D, CL>(a, smem, ms, bh, h, row0, nch, rank);
  } else if (warp < 8) {
    role_operands<D, CL>(a, smem, ms, h, row0, nch, rank);
  } else if (warp < 12) {
    role_epilogue<D, CL, LN>(a, smem, ms, bh, row0, nch);
  } else if (warp == 12) {
    if ((threadIdx.x & 31) == 0) role_mma<D, CL>(a, smem, ms, nch);
  } else if ((threadIdx.x & 31) == 0) {
    role_tma<D, CL>(p, smem, ms, bh, nch, rank);
  } else if ((threadIdx.x & 31) == 1) {
    role_tma_u<D, CL>(p, smem, ms, bh, nch, rank);
  } else if (CL > 1 && (threadIdx.x & 31) == 2) {
    role_wdone_observer<CL>(a, ms, nch);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    // every MMA has completed once `fin` fires (it is committed after the last one)
    if (!mbar_wait(&ms->fin, 0, &ms->never, 4000000000ull)) report(a.status, kErrTimeout);
    tc_fence_after();
    tmem_dealloc(ms->tmem, 512);
  }
  if (CL > 1 && threadIdx.x == 0 && nch > 0) {
    // The other CTA's last stage and weight releases land in this CTA's barriers: wait for
    // them (bounded) so that no arrival targets this CTA after it exits.  Every earlier phase
    // of these barriers was waited for in order, so the parity identifies the phase.
    for (int st = 0; st < CF::NSQ && st < nch; ++st) {
      const int c_last = st + ((nch - 1 - st) / CF::NSQ) * CF::NSQ;
      if (!mbar_wait_cl(&ms->qk_empty[st], (c_last / CF::NSQ) & 1, &ms->never, 1ll << 31))
        report(a.status, kErrTimeout);
    }
    // (every phase of w_done was waited for by the observer thread before the final barrier)
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
  constexpr int kClY = LN ? D / kDV : kCL;
  static_assert(!LN || kCL == 1, "the LayerNorm cluster spans the value slices");
  static std::atomic<uint64_t> attr_set{0};  // bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(chunk_kernel<D, kCL, LN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Cfg<D, kCL>::SMEM);
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
  static_assert((D / kDV) % kCL == 0, "value slices pair up into clusters");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(BH, D / kDV, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg<D, kCL>::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = kClY;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kClY > 1 ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, chunk_kernel<D, kCL, LN>, p);
  count_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool chunk_supported(int d, int dtype, int causal) {
  return dtype == 0 && causal == 1 && (d == 64 || d == 128);
}

cudaError_t launch_fwd_chunk(const FwdArgs& a, cudaStream_t stream) {
  if (a.d == 64) return a.ln ? launch_d<64, true>(a, stream) : launch_d<64, false>(a, stream);
  if (a.d == 128) return a.ln ? launch_d<128, true>(a, stream) : launch_d<128, false>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace zs
