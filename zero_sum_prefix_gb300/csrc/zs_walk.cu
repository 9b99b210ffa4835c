// Causal ZeroS forward for d = 64, bf16 inputs: one CTA per (sequence, segment) that owns all
// 64 value columns of its head, on the tensor cores (tcgen05 / TMEM / TMA).
//
// Method: Paper-Notes "ZeroS: Zero-Sum Linear Attention for Efficient Transformers", method
// details: deviation logits, zero-sum weights w_{t,i} = sig1_t delta_{t,i}/t + sigh_t eps_{t,i},
// angular factor q_hat_t R_{t-i} k_hat_i^T, and the "linear-time prefix scan" whose five states
// (E, P, F, G, H) give o_t = q_hat_t (alpha_t F_t + beta_t G_t + gamma_t H_t).
//
// Chunked form (chunks of C = 128 tokens).  With the chunk reference M_c (the running maximum of
// s at the chunk's last token), Q = unit(rot(q)) and K = unit(rot(k)), the row coefficients
// (a, b, g)_t = (sigh_t e^{M_c - m_t} / Et_t, beta_t, gamma_t) and the column scalars
// (e_i, s_i) = (e^{s_i - M_c}, s_i):
//     W_{t,i} = a_t e_i + b_t s_i + g_t                (fp32 on the CUDA cores)
//     S_{t,i} = [i <= t] (Q_t . K_i) W_{t,i}           (fp32 product, rounded once to fp16)
//     X = Q [F~ | G | H]  (state before the chunk, fp16 copy),   X_SV = S V
//     o_t = X_SV + a_t X_F + b_t X_G + g_t X_H
//     state^T += [e v | s v]^T K  and  [v | e v]^T K    (F~ rescaled by e^{M_{c-1} - M_c} first)
// The weight is formed in fp32 before the product is rounded: its three terms nearly cancel
// (the weights of a query sum to zero).  The scalars s, m, Et = E e^{-m}, P of every token come
// from the scalar pass (zs_scalars.cu, the canonical blocked fp32 order), which runs first; this
// kernel is launched as its programmatic dependent, so it sets up its barriers and tensor memory
// while the pass ends and waits for the pass (grid_dep_wait) before any role starts.
//
// Operand precision.  Every tensor-core operand is fp16 (fp32 accumulation): the unit vectors,
// S and the value-side tiles have 11 significant bits instead of bf16's 8, which is what the
// error of short sequences is made of.  The range is kept by exact powers of two folded into
// the fp32 coefficients: row t of S carries 2^kr_t (|S| < 1), the state copy feeding chunk c
// carries 2^-kb_c (2^kb_c > 128 c, the number of tokens it sums), and G is carried with
// s 2^-ks (|s 2^-ks| < 1 over the sequence, from the scalar pass).  The copy's F~ is kept at the
// running maximum before the chunk (its largest factor e^{s - m} is then 1, away from fp16's
// subnormals), the output coefficient of X_F taking the chunk's e^{m - M_c}.  Values must lie
// within the fp16 range (|v| <= 65504, reported otherwise).
//
// Split along the sequence.  When the sequences are fewer than the SMs, each is cut into
// segments; the CTA of a later segment first replays the state side of the chunks before its
// segment (rotated unit keys, scaled values and the state products, with one fixed reference,
// the running maximum at the token before the segment) and then walks its own chunks.  No CTA
// waits for another, and the replay costs a fraction of a full chunk (no queries, no intra-chunk
// products, no outputs), so the segment lengths are chosen geometric to equalise the CTAs.
//
// Warp roles (576 threads, one CTA per SM):
//   warps 0-7   (O) : operands; token row r = 16 w + lane / 2, half hf = lane & 1 of the row's
//                     rotary pairs: norms (halves exchanged by a shuffle), rotation and unit
//                     scaling of q and k in place (TMA-landed tiles), column scalars (hf = 0),
//                     row coefficients (hf = 1), half of the row's value-side tiles.
//   warps 8-15  (E) : two per TMEM lane quadrant: S tile from Q K^T, the state copy after each
//                     update (TMEM -> fp16 B tile of the next chunk's Q [F~|G|H] product, and the
//                     F~ rescale in TMEM), output rows from X (staged in shared memory, one TMA
//                     store per chunk), the final state (prefill).
//   warp 16     (M) : TMEM allocation; the whole warp runs the issue loop (warp-uniform
//                     operands) and one elected lane issues every tcgen05.mma.
//   warp 17     (T) : TMA producer of q, k, v (three stages), with L2 prefetch ahead.
// The fused output LayerNorm is not done here: it runs on the chunked kernel of zs_chunk.cu,
// whose value slices exchange row statistics in a cluster (measured faster than whole rows
// per thread with one E warp per quadrant here: 0.155 against 0.169 ms per call at
// B8 H8 N4096).
// TMEM (512 columns): [0,128) Q K^T (the fp16 S tile overlays it: K step h in [16 h, 16 h + 8)),
// [128,320) X = Q[F~|G|H],
// [320,384) X_SV, [384,448) state A = [F~^T ; G^T], [448,512) state B = [H^T ; F~^T].
// The state B accumulator repeats F~^T in its upper lanes so that every copy warp reads 96
// columns: quadrants 0/1 take F~ columns 0-31 from A and H from B, quadrants 2/3 G from A and
// F~ columns 32-63 from B (each half of F~ is rescaled where it is read).
// Every mbarrier wait is bounded; a timeout records ZEROS_ERR_TIMEOUT, raises a CTA abort flag
// and every role leaves its loop; TMA loads in flight are waited for and TMEM is released after
// the last MMA completes.
#include <math.h>

#include <atomic>

#include "zs_common.cuh"
#include "zs_internal.h"
#include "zs_range.cuh"
#include "zs_sm100.cuh"

namespace zs {
namespace {

using namespace sm100;

constexpr int kC = 128;                 // tokens per chunk
constexpr int kD = 64;                  // head dimension
constexpr uint32_t kTile = 128 * 128;   // one 16-bit [128 x 64] atom tile (128 rows of 128 bytes)
constexpr int kNST = 3;                 // q/k/v stages
constexpr int kOpWarps = 8;
constexpr int kEpWarp0 = 8;             // from warp 8: S tiles, state copies, outputs
constexpr int kEpq = 2;                 // E warps per TMEM lane quadrant (they split every E task)
constexpr int kMmaWarp = kEpWarp0 + 4 * kEpq;
constexpr int kThreads = (kMmaWarp + 2) * 32;
constexpr int kMaxSeg = 4;

struct WLay {
  static constexpr uint32_t Q = 0;
  static constexpr uint32_t K = Q + kNST * kTile;
  static constexpr uint32_t V = K + kNST * kTile;
  static constexpr uint32_t VSC = V + kNST * kTile;       // 2 atoms: e v | s v
  static constexpr uint32_t SB = VSC + 2 * kTile;         // state B tile: 192 rows x 128 bytes
  static constexpr uint32_t OUTS = SB + 192 * 128;        // output staging, [128 x 64] bf16
  static constexpr uint32_t COL = OUTS + kTile;           // float2 [stage][128]: (e_i, s_i)
  static constexpr uint32_t COEF = COL + kNST * kC * 8;   // float4 [stage][128], the row scales:
                                                          // (a, b 2^(kb+ks), g 2^kb, 2^kr)
  static constexpr uint32_t THETA = COEF + kNST * kC * 16;  // float [32]: rotary frequencies
  static constexpr uint32_t PHI = THETA + 128;            // float [stage][32]: chunk base angles
  static constexpr uint32_t MISC = PHI + kNST * 128;
  static constexpr uint32_t BYTES = MISC + 512;
};
static_assert(WLay::BYTES <= 232448, "shared memory budget of one CTA");
static_assert(WLay::SB % 1024 == 0 && WLay::OUTS % 1024 == 0, "swizzled tiles are 1 KB aligned");

constexpr uint32_t TM_A = 0, TM_X = 128, TM_SV = 320, TM_SA = 384, TM_SBS = 448;

struct WMisc {
  uint64_t full[kNST];   // q, k, v of a stage landed (TMA transaction count)
  uint64_t empty[kNST];  // the stage's tiles consumed by the MMAs
  uint64_t opd[kNST];    // operand warps done: Q, K rotated, coefficients, columns, scaled values
  uint64_t vsc_free;     // the previous state update has read the scaled values
  uint64_t a_full, s_full, x_full, x_free;
  uint64_t u_done;       // a state update completed (the next chunk needs a copy)
  uint64_t st_done;      // the copy read the state (F~ rescaled in TMEM) and wrote the B tile
  uint64_t sb_free;      // the Q [F~|G|H] product has read the B tile
  uint64_t ob_free;      // the output staging tile may be written (previous store has read it)
  uint64_t ob_full;      // the output staging tile is written (the store may start)
  uint64_t fin;          // every MMA has completed
  uint32_t tmem;
  int abort;
  int never;             // stays 0: lets the final waits ignore the abort flag
};
static_assert(sizeof(WMisc) <= 512, "WMisc fits its shared-memory slot");

struct WalkParams {
  CUtensorMap tq, tk, tv, to;  // [B*H, N, 64] bf16, box {64, 128, 1}, 128-byte swizzle
  FwdArgs a;
  const float* ang;            // rope: theta[32], then phi[nch][32] (chunk base angles mod 2 pi)
  int nseg;                    // segments per sequence
  int seg_start[kMaxSeg + 1];  // segment j covers chunks [seg_start[j], seg_start[j + 1])
  long long wait_limit;        // bound of every wait, SM clock cycles
  int dbg_skip;                // testing hook: one warp withholds its first S-tile arrival
};

__device__ __forceinline__ void fail_wait(WMisc* ms, int* status) {
  report(status, kErrTimeout);
  ms->abort = 1;
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) global -> shared,
// completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// The scalar pass's output is read through L2 only (ld.global.cg): this kernel is launched as a
// programmatic dependent of that pass and may start while it still writes the buffer, so no read
// may be served from a line cached before its grid_dep_wait().
__device__ __forceinline__ float4 scal_at(const float4* scal, int i) { return __ldcg(scal + i); }

// Running maximum at the last token of chunk c (the chunk reference M_c).
__device__ __forceinline__ float chunk_ref(const float4* scal, int c, int N) {
  return scal_at(scal, min(N, (c + 1) * kC) - 1).y;
}

// Scale exponent of the state copy that feeds chunk c's Q [F~|G|H] product.
__device__ __forceinline__ int state_exp(int c) { return zs::state_exp(c, kC); }

// ============================================================================ T: TMA producer
// Per chunk: q (walk chunks), k, v into the chunk's stage, and the chunk's rotary base angles
// (128 bytes of the angle table) with them; the chunks two and three ahead are prefetched into
// L2 while the stages are in use.
__device__ void role_tma(const WalkParams& p, uint8_t* smem, WMisc* ms, int bh, int c0, int c1) {
  const uint32_t base = smem_u32(smem);
  const long long lim = p.wait_limit;
  const bool rope = p.a.rope != 0;
  tma_prefetch_desc(&p.tq);
  tma_prefetch_desc(&p.tk);
  tma_prefetch_desc(&p.tv);
  auto prefetch = [&](int cc) {
    if (cc < c1) {
      if (cc >= c0) tma_prefetch_3d(&p.tq, 0, cc * kC, bh);
      tma_prefetch_3d(&p.tk, 0, cc * kC, bh);
      tma_prefetch_3d(&p.tv, 0, cc * kC, bh);
    }
  };
  prefetch(kNST);
  prefetch(kNST + 1);
  int issued = 0;  // chunks whose loads were issued
  bool ok = true;
  for (int c = 0; c < c1; ++c) {
    const int st = c % kNST;
    if (c >= kNST &&
        !mbar_wait(&ms->empty[st], (uint32_t)((c / kNST) - 1) & 1u, &ms->abort, lim)) {
      ok = false;
      break;
    }
    const bool walk = c >= c0;
    uint64_t* fb = &ms->full[st];
    mbar_arrive_expect_tx(fb, (walk ? 3u : 2u) * kTile + (rope ? 128u : 0u));
    if (walk) tma_load_3d(base + WLay::Q + st * kTile, &p.tq, 0, c * kC, bh, fb);
    tma_load_3d(base + WLay::K + st * kTile, &p.tk, 0, c * kC, bh, fb);
    tma_load_3d(base + WLay::V + st * kTile, &p.tv, 0, c * kC, bh, fb);
    if (rope) bulk_load(base + WLay::PHI + st * 128, p.ang + 32 + (size_t)c * 32, 128, fb);
    issued = c + 1;
    prefetch(c + kNST + 2);
  }
  if (!ok) fail_wait(ms, p.a.status);
  // never leave with copies in flight into this CTA's shared memory: wait for the last loads
  // of every stage (a wait on a phase that already completed returns at once)
  for (int c = max(0, issued - kNST); c < issued; ++c)
    mbar_wait(&ms->full[c % kNST], (uint32_t)(c / kNST) & 1u, &ms->never, lim);
}

// ============================================================================ O: operands
// Shared-memory chunk of slot s (0..3) of a thread's half row: half 0 takes the 16-byte chunks
// {0, 4, 1, 5}, half 1 {6, 2, 7, 3}, so that the two halves of four consecutive rows hit eight
// different bank groups in every access.  Slot s holds first elements of rotary pairs
// (columns < 32) when ((s & 1) ^ hf) == 0, else their partners (columns + 32).
__device__ __forceinline__ int op_chunk(int s, int hf) {
  return ((((s & 1) ^ hf)) << 2) + 2 * hf + (s >> 1);
}

struct RowIn {  // per-token inputs of a row, loaded one chunk ahead
  float4 sc;    // (s, m, Et, P)
  float M;      // chunk reference
  float x1, xh, x0;
};

// Rotate (RoPE) and scale one group of 8 rotary pairs of bf16 inputs: pair (xa, xb) ->
// f (xa cos - xb sin, xa sin + xb cos), written as fp16 (unit vectors: in range, and eight times
// finer than bf16); cs[k] = (cos, sin) of the pair's angle.
__device__ __forceinline__ void rot_group(uint4& wa, uint4& wb, const float2 (&cs)[8], float f,
                                          bool rope) {
  const uint32_t ia[4] = {wa.x, wa.y, wa.z, wa.w}, ib[4] = {wb.x, wb.y, wb.z, wb.w};
  uint32_t oa[4], ob[4];
  const float2 f2 = make_float2(f, f);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float2 xa, xb;
    unpack_bf16x2(ia[k], xa.x, xa.y);
    unpack_bf16x2(ib[k], xb.x, xb.y);
    float2 na, nb;
    if (rope) {
      const float2 c2 = __fmul2_rn(make_float2(cs[2 * k].x, cs[2 * k + 1].x), f2);
      const float2 s2 = __fmul2_rn(make_float2(cs[2 * k].y, cs[2 * k + 1].y), f2);
      na = __ffma2_rn(xa, c2, __fmul2_rn(make_float2(-xb.x, -xb.y), s2));
      nb = __ffma2_rn(xa, s2, __fmul2_rn(xb, c2));
    } else {
      na = __fmul2_rn(xa, f2);
      nb = __fmul2_rn(xb, f2);
    }
    oa[k] = pack_f16x2(na.x, na.y);
    ob[k] = pack_f16x2(nb.x, nb.y);
  }
  wa = make_uint4(oa[0], oa[1], oa[2], oa[3]);
  wb = make_uint4(ob[0], ob[1], ob[2], ob[3]);
}

__device__ __forceinline__ float sumsq_words(const uint4 (&w)[4]) {
  float2 ss = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const uint32_t ws[4] = {w[s].x, w[s].y, w[s].z, w[s].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 x;
      unpack_bf16x2(ws[k], x.x, x.y);
      ss = __ffma2_rn(x, x, ss);
    }
  }
  return ss.x + ss.y;
}

__device__ void role_op(const WalkParams& p, uint8_t* smem, WMisc* ms, int bh, int c0, int c1) {
  const FwdArgs& a = p.a;
  const long long lim = p.wait_limit;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hf = lane & 1;
  const int r = 16 * warp + (lane >> 1);  // token row inside the chunk
  const int N = a.N;
  const size_t row0 = (size_t)bh * N;
  const float4* scal = a.scal + row0;
  const uint32_t base = smem_u32(smem);
  const bool rope = a.rope != 0;
  // rotary frequencies of this half's 16 pairs (pairs 16 hf .. 16 hf + 15), in shared memory
  const uint32_t th_s = base + WLay::THETA + 64 * hf;
  const float M_ref = c0 > 0 ? scal_at(scal, c0 * kC - 1).y : 0.0f;  // replay reference
  const int ks = s_exp(a, bh);
  const float sinv = pow2f(-ks);
  const float smax_seq = seq_smax(a, bh);  // the sequence's largest |s| (bounds a row's weights)

  auto load_in = [&](int cc) {
    RowIn o{make_float4(0.f, 0.f, 0.f, 0.f), 0.0f, 0.0f, 0.0f, -INFINITY};
    if (cc < c1) {
      o.M = cc >= c0 ? chunk_ref(scal, cc, N) : M_ref;
      const int i = cc * kC + r;
      if (i < N) {
        o.sc = scal_at(scal, i);
        if (cc >= c0 && hf == 1) {
          o.x1 = a.g1[row0 + i];
          o.xh = a.gh[row0 + i];
          if (a.g0) o.x0 = a.g0[row0 + i];
        }
      }
    }
    return o;
  };
  RowIn cur = load_in(0);

  for (int c = 0; c < c1; ++c) {
    const int st = c % kNST;
    const bool walk = c >= c0;
    const int i = c * kC + r;
    const bool valid = i < N;
    if (!mbar_wait_warp_lim(&ms->full[st], (uint32_t)(c / kNST) & 1u, &ms->abort, lim)) {
      fail_wait(ms, a.status);
      return;
    }
    const RowIn nxt = load_in(c + 1);
    const uint32_t ph_s = base + WLay::PHI + st * 128 + 64 * hf;
    const uint32_t qt = base + WLay::Q + st * kTile, kt = base + WLay::K + st * kTile;
    const uint32_t vt = base + WLay::V + st * kTile, vs = base + WLay::VSC;
    // ---- unit rotated keys (and queries in walk chunks), in place ----
    uint4 kw[4], qw[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) kw[s] = lds128(kt + sw128_off(r, op_chunk(s, hf)));
    if (walk) {
#pragma unroll
      for (int s = 0; s < 4; ++s) qw[s] = lds128(qt + sw128_off(r, op_chunk(s, hf)));
    }
    float kk = sumsq_words(kw);
    kk += __shfl_xor_sync(0xffffffffu, kk, 1);
    const float kap = rsqrtf(fmaxf(kk, 1e-24f));
    float rho = 0.0f;
    if (walk) {
      float qq = sumsq_words(qw);
      qq += __shfl_xor_sync(0xffffffffu, qq, 1);
      rho = rsqrtf(fmaxf(qq, 1e-24f));
    }
    const float rf = (float)r;
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      float2 cs[8];
      if (rope) {
        // this group's 8 frequencies and chunk base angles, as 16-byte shared loads
        const float4 t0 = lds128f(th_s + 32 * g), t1 = lds128f(th_s + 32 * g + 16);
        const float4 f0 = lds128f(ph_s + 32 * g), f1 = lds128f(ph_s + 32 * g + 16);
        const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
        const float fv[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          float sn, cn;
          __sincosf(__fmaf_rn(rf, tv[k], fv[k]), &sn, &cn);
          cs[k] = make_float2(cn, sn);
        }
      }
      // slots 2g and 2g + 1 hold the pairs' first elements and their partners, in an order
      // set by the half (selected by value: a register array indexed by a runtime value would
      // live in local memory)
      uint4 ka = hf ? kw[2 * g + 1] : kw[2 * g], kb = hf ? kw[2 * g] : kw[2 * g + 1];
      rot_group(ka, kb, cs, kap, rope);
      kw[2 * g] = hf ? kb : ka;
      kw[2 * g + 1] = hf ? ka : kb;
      if (walk) {
        uint4 qa = hf ? qw[2 * g + 1] : qw[2 * g], qb = hf ? qw[2 * g] : qw[2 * g + 1];
        rot_group(qa, qb, cs, rho, rope);
        qw[2 * g] = hf ? qb : qa;
        qw[2 * g + 1] = hf ? qa : qb;
      }
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) sts128(kt + sw128_off(r, op_chunk(s, hf)), kw[s]);
    if (walk) {
#pragma unroll
      for (int s = 0; s < 4; ++s) sts128(qt + sw128_off(r, op_chunk(s, hf)), qw[s]);
    }
    // ---- column scalars (e_i, s_i) and row coefficients (a, b, g) ----
    const float s_i = cur.sc.x, M = cur.M;
    float ce = 0.0f, cs1 = 0.0f;
    if (valid) {
      ce = __expf(s_i - M);
      cs1 = s_i;
      if (!isfinite(ce)) report(a.status, kErrRange);
    }
    if (walk) {
      if (hf == 0) {
        sts64f(base + WLay::COL + (st * kC + r) * 8, ce, cs1);
      } else {
        // a as the S tile uses it (reference M_c), (b, g) scaled by 2^kb (the state copy's
        // scale) and b also by 2^ks (G is carried with s 2^-ks), and the row's S scale 2^kr with
        // |S| 2^kr < 1: |W| <= |a| + |b| max|s| + |g|
        float4 cf = make_float4(0.f, 0.f, 0.f, 1.f);
        if (valid) {
          const float m = cur.sc.y, Et = cur.sc.z, P = cur.sc.w;
          const float sig1 = __fdividef(1.0f, 1.0f + __expf(-cur.x1));
          const float sigh = __fdividef(1.0f, 1.0f + __expf(-cur.xh));
          const float rt = __fdividef(1.0f, (float)(i + 1));
          const float bc = (sig1 - sigh) * rt;
          float ca = __fdividef(sigh, Et) * __expf(M - m);
          float cg = -(bc * P * rt + sigh * rt);
          if (a.g0) cg += __fdividef(1.0f, 1.0f + __expf(-cur.x0)) * rt;  // zero-order gate
          if (!isfinite(ca)) report(a.status, kErrRange);
          // a e_i over the row's keys i <= t is at most sigma^h / E~ (e^{s_i - m_t} <= 1)
          const int kb = state_exp(c);
          const int kr = row_exp(__fdividef(sigh, Et) + fabsf(bc) * smax_seq + fabsf(cg));
          cf = make_float4(ca, bc * pow2f(kb + ks), cg * pow2f(kb), pow2f(kr));
        }
        sts128f(base + WLay::COEF + (st * kC + r) * 16, cf);
      }
    }
    // ---- half of the row's scaled values: columns 32 hf .. 32 hf + 31 (single buffer: the
    //      previous state update must have read it) ----
    if (c >= 1 && !mbar_wait_warp_lim(&ms->vsc_free, (uint32_t)(c - 1) & 1u, &ms->abort, lim)) {
      fail_wait(ms, a.status);
      return;
    }
    {
      // the value tile becomes fp16 in place (exact for bf16 values within the fp16 range;
      // larger ones are reported), with e v and (s 2^-ks) v beside it
      const float2 e2 = make_float2(ce, ce), s2 = make_float2(cs1 * sinv, cs1 * sinv);
      uint32_t vmax = 0u;  // largest |v| of the row's half, as bf16 pairs
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint32_t off = sw128_off(r, 4 * hf + s);
        const uint4 wv = lds128(vt + off);
        const uint32_t pv[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t ph[4], pe[4], ps[4];
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          float2 v2;
          unpack_bf16x2(pv[y], v2.x, v2.y);
          vmax = bf16x2_absmax(vmax, pv[y]);
          const float2 ev = __fmul2_rn(e2, v2), sv = __fmul2_rn(s2, v2);
          ph[y] = pack_f16x2(v2.x, v2.y);
          pe[y] = pack_f16x2(ev.x, ev.y);
          ps[y] = pack_f16x2(sv.x, sv.y);
        }
        sts128(vt + off, make_uint4(ph[0], ph[1], ph[2], ph[3]));
        sts128(vs + off, make_uint4(pe[0], pe[1], pe[2], pe[3]));
        sts128(vs + kTile + off, make_uint4(ps[0], ps[1], ps[2], ps[3]));
      }
      // bf16 values from 65536 up (and inf, NaN) are beyond the fp16 range
      if ((vmax & 0xffffu) >= 0x4780u || (vmax >> 16) >= 0x4780u) report(a.status, kErrRange);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ms->opd[st]);
    cur = nxt;
  }
}

// ============================================================================ M: MMA issue
// Per chunk c, in issue order:
//   A = Q K^T                          (walk chunks; Q, K rotated)                  -> a_full
//   state += [e v | s v]^T K, [v | e v]^T K   (the copy read the previous state)    -> u_done
//   X = Q [F~ | G | H]                 (walk chunks after the first; B tile written,
//                                       previous outputs read)                      -> sb_free
//   X_SV = S V                         (walk chunks; S tile formed)                 -> x_full
//   stage released                                                                  -> empty
// MMAs issued by this thread execute in order, so A of a chunk may overwrite the S tile that
// the previous chunk's S V product reads.  The whole warp runs this loop (its operands stay
// warp-uniform, so the issue stays short next to the busy warps of the same scheduler) and one
// elected lane issues.
__device__ void role_mma(const WalkParams& p, uint8_t* smem, WMisc* ms, int c0, int c1) {
  const bool leader = elect_one();
  const uint32_t base = smem_u32(smem);
  const uint32_t tm = ms->tmem;
  const long long lim = p.wait_limit;
  constexpr uint32_t id_qk = idesc_f16_f32(128, 128, false, false);
  constexpr uint32_t id_x = idesc_f16_f32(128, 192, false, false);
  constexpr uint32_t id_u = idesc_f16_f32(128, kD, true, true);
  constexpr uint32_t id_sv = idesc_f16_f32(128, kD, false, true);
  // descriptors: the start address field is address / 16, and every tile lies below 256 KB,
  // so the descriptor of base + off is the base's descriptor + off / 16
  const uint64_t dq = sw128_desc(base + WLay::Q, 16, 1024);
  const uint64_t dk = sw128_desc(base + WLay::K, 16, 1024);
  const uint64_t dkm = sw128_desc(base + WLay::K, kTile, 1024);     // K as MN-major B
  const uint64_t dvsc = sw128_desc(base + WLay::VSC, kTile, 1024);  // [e v | s v], MN-major A
  const uint64_t dvb = sw128_desc(base + WLay::V, kTile, 1024);     // V as MN-major B
  const uint64_t dsb = sw128_desc(base + WLay::SB, 16, 1024);       // [F~|G|H] K-major B
  const int cfirst = c0 > 0 ? c0 - 1 : 0;  // first update followed by a state copy
  bool ok = true;
  for (int c = 0; c < c1; ++c) {
    const int st = c % kNST;
    const bool walk = c >= c0;
    const int wi = c - c0;
    const uint64_t so = (uint64_t)((st * kTile) >> 4);
    if (!mbar_wait_warp_lim(&ms->opd[st], (uint32_t)(c / kNST) & 1u, &ms->abort, lim)) {
      ok = false;
      break;
    }
    tc_fence_after();
    if (walk && leader) {
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        const uint64_t off = (uint64_t)((kk * 32) >> 4);
        mma_f16kind(tm + TM_A, dq + so + off, dk + so + off, id_qk, kk > 0);
      }
      mma_commit(&ms->a_full);
    }
    __syncwarp();
    // ---- state update (M = 128 value rows, N = 64 key columns, K = the chunk's tokens) ----
    if (c >= 1 && c - 1 >= cfirst) {
      if (!mbar_wait_warp_lim(&ms->st_done, (uint32_t)(c - 1 - cfirst) & 1u, &ms->abort, lim)) {
        ok = false;
        break;
      }
      tc_fence_after();
    }
    if (leader) {
      const uint32_t va = base + WLay::V + st * kTile;
      const uint32_t lbo = (base + WLay::VSC) - va;  // [v | e v]: the second atom is e v
      const uint64_t dva = sw128_desc(va, lbo, 1024);
#pragma unroll
      for (int kk = 0; kk < kC / 16; ++kk) {
        const uint64_t off = (uint64_t)((kk * 2048) >> 4);
        const uint32_t acc = (c > 0 || kk > 0) ? 1u : 0u;
        mma_f16kind(tm + TM_SA, dvsc + off, dkm + so + off, id_u, acc);
        mma_f16kind(tm + TM_SBS, dva + off, dkm + so + off, id_u, acc);
      }
      mma_commit(&ms->vsc_free);
      if (c >= cfirst && c <= c1 - 2) mma_commit(&ms->u_done);
    }
    __syncwarp();
    if (walk) {
      if (c > 0) {
        // ---- X = Q [F~ | G | H] with the state before this chunk (its copy was waited for
        //      before the state update) ----
        if (wi >= 1 &&
            !mbar_wait_warp_lim(&ms->x_free, (uint32_t)(wi - 1) & 1u, &ms->abort, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint64_t off = (uint64_t)((kk * 32) >> 4);
            mma_f16kind(tm + TM_X, dq + so + off, dsb + off, id_x, kk > 0);
          }
          mma_commit(&ms->sb_free);
        }
        __syncwarp();
      } else if (wi >= 1 &&
                 !mbar_wait_warp_lim(&ms->x_free, (uint32_t)(wi - 1) & 1u, &ms->abort, lim)) {
        ok = false;
        break;
      }
      // ---- X_SV = S V (S from TMEM) ----
      if (!mbar_wait_warp_lim(&ms->s_full, (uint32_t)wi & 1u, &ms->abort, lim)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk) {
          const uint64_t boff = (uint64_t)((kk * 2048) >> 4);  // MN-major B, 16 token rows/step
          mma_f16kind_ts(tm + TM_SV, tm + TM_A + kk * 16, dvb + so + boff, id_sv, kk > 0);
        }
        mma_commit(&ms->x_full);
      }
      __syncwarp();
    }
    if (leader) mma_commit(&ms->empty[st]);
    __syncwarp();
  }
  if (leader) {
    if (!ok) fail_wait(ms, p.a.status);
    mma_commit(&ms->fin);
  }
  __syncwarp();
}

// ============================================================================ E: S tiles,
// state copies and outputs.  Warp w & 3 owns TMEM lane quadrant w & 3.  Per walk chunk c, in
// order: the S tile of c (after Q K^T), the state copy after the update of c (for the next
// chunk's Q [F~|G|H] product), then the output rows of c (after S V).  The copy after the last
// replayed update comes before the first walk chunk.
//
// State copy: lane L of quadrant wq reads 96 state columns (three 32-column pieces):
//   wq 0/1 (j = L):      A[0:32] = F~ row j cols 0-31,  B[0:32], B[32:64] = H row j
//   wq 2/3 (j = L - 64): A[0:32], A[32:64] = G row j,   B[32:64] = F~ row j cols 32-63
// and writes them as fp16 into the B tile rows (F~: j, G: 64 + j, H: 128 + j).  (Giving
// quadrants 2/3, whose S tiles are the largest, a smaller share of the copy measured slower:
// the update after the copy waits for the slowest warp.)
struct Piece {
  uint32_t col;  // TMEM column offset
  int row;       // B tile row
  int ch0;       // first 16-byte chunk
  bool f;        // F~ (rescaled)
  int rec;       // record matrix: 0 F~, 1 G, 2 H
  int a0;        // first key column
};

constexpr int kStPieces = 3;  // 32-column pieces of the state copied per lane
__device__ __forceinline__ Piece st_piece(int wq, int L, int k) {
  const bool lo = wq < 2;
  const int j = lo ? L : L - 64;
  if (lo) {
    if (k == 0) return Piece{TM_SA, j, 0, true, 0, 0};
    return Piece{TM_SBS + 32u * (k - 1), 128 + j, 4 * (k - 1), false, 2, 32 * (k - 1)};
  }
  if (k < 2) return Piece{TM_SA + 32u * k, 64 + j, 4 * k, false, 1, 32 * k};
  return Piece{TM_SBS + 32u, j, 4, true, 0, 32};
}

// The copy after the update of chunk c (copy index k = c - cfirst): the fp16 B tile (times
// 2^-kb) keeps F~ at its reference M_cur, the running maximum at the state's last token (so that
// the largest of its factors e^{s - M_cur} is 1 and fp16 keeps its digits), while F~ in TMEM is
// rescaled to the next chunk's reference M_next for the next update.  It first waits until
// the Q [F~|G|H] product of chunk c has read the B tile; that product was issued right after
// the update and the next update queues behind it on the tensor pipe, so the wait costs no
// tensor time.  Returns false when a wait gave up.
template <int EPQ>
__device__ __forceinline__ bool state_copy(WMisc* ms, uint32_t tm, uint32_t base, int wq, int hb,
                                           int L, int c, int k, int xfirst, float M_cur,
                                           float M_next, long long lim) {
  const bool resc = M_next > M_cur;
  const float fac = resc ? expf(M_cur - M_next) : 1.0f;
  const float sc = pow2f(-state_exp(c + 1));  // fp16 range of the next chunk's B tile
  if (!mbar_wait_warp_lim(&ms->u_done, (uint32_t)k & 1u, &ms->abort, lim)) return false;
  if (c >= xfirst &&
      !mbar_wait_warp_lim(&ms->sb_free, (uint32_t)(c - xfirst) & 1u, &ms->abort, lim))
    return false;
  tc_fence_after();
  // each of the EPQ warps of the quadrant copies 32 / EPQ columns of every piece
  constexpr int W = 32 / EPQ;
  auto put = [&](const Piece& pc, uint32_t (&v)[W]) {
    const float2 sc2 = make_float2(sc, sc);
#pragma unroll
    for (int x = 0; x < W / 8; ++x) {
      const uint32_t* w8 = v + 8 * x;
      uint32_t pk[4];
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const float2 f = __fmul2_rn(make_float2(__uint_as_float(w8[2 * y]),
                                                __uint_as_float(w8[2 * y + 1])), sc2);
        pk[y] = pack_f16x2(f.x, f.y);
      }
      sts128(base + WLay::SB + sw128_off(pc.row, pc.ch0 + (W / 8) * hb + x),
             make_uint4(pk[0], pk[1], pk[2], pk[3]));
    }
    if (pc.f && resc) {
      const float2 f2 = make_float2(fac, fac);
#pragma unroll
      for (int y = 0; y < W; y += 2) {
        const float2 f = __fmul2_rn(make_float2(__uint_as_float(v[y]), __uint_as_float(v[y + 1])), f2);
        v[y] = __float_as_uint(f.x);
        v[y + 1] = __float_as_uint(f.y);
      }
      if constexpr (EPQ == 1) tmem_st32_nowait(tm + pc.col, v);
      else tmem_st16_nowait(tm + pc.col + W * hb, v);
    }
  };
  auto ld = [&](const Piece& pc, uint32_t (&v)[W]) {
    if constexpr (EPQ == 1) tmem_ld32_nowait(tm + pc.col, v);
    else tmem_ld16_nowait(tm + pc.col + W * hb, v);
  };
  {
    const Piece p0 = st_piece(wq, L, 0), p1 = st_piece(wq, L, 1);
    uint32_t v0[W], v1[W];
    ld(p0, v0);
    ld(p1, v1);
    tmem_wait_ld();
    reg_fence(v0);
    reg_fence(v1);
    put(p0, v0);
    put(p1, v1);
  }
  {
    const Piece p2 = st_piece(wq, L, 2);
    uint32_t v2[W];
    ld(p2, v2);
    tmem_wait_ld();
    reg_fence(v2);
    put(p2, v2);
  }
  tmem_wait_st();
  tc_fence_before();
  fence_proxy_async_smem();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&ms->st_done);
  return true;
}

__device__ void role_e(const WalkParams& p, uint8_t* smem, WMisc* ms, int bh, int c0, int c1) {
  constexpr int EPQ = kEpq;
  const FwdArgs& a = p.a;
  const long long lim = p.wait_limit;
  const int wq = (threadIdx.x >> 5) & 3;       // TMEM lane quadrant of this warp
  const int hb = ((threadIdx.x >> 5) - kEpWarp0) >> 2;  // which of the quadrant's E warps
  const int t = wq * 32 + (threadIdx.x & 31);  // TMEM lane = token row (S, outputs)
  const uint32_t tm = ms->tmem + ((uint32_t)(wq * 32) << 16);
  const uint32_t base = smem_u32(smem);
  const bool leader = threadIdx.x == kEpWarp0 * 32;
  const int N = a.N;
  const float4* scal = a.scal + (size_t)bh * N;
  const float sinv = pow2f(-s_exp(a, bh));  // G is carried with s 2^-ks
  const int cfirst = c0 > 0 ? c0 - 1 : 0;  // first update followed by a state copy
  const int xfirst = max(c0, 1);           // first chunk with a Q [F~|G|H] product
  // chunk references of the current and the next chunk, loaded one chunk ahead
  float Mc = chunk_ref(scal, c0, N);
  float Mn = c0 + 1 < c1 ? chunk_ref(scal, c0 + 1, N) : 0.0f;
  // the running maximum at the token before the current chunk (the B tile's F~ reference)
  float Mp = c0 > 0 ? scal_at(scal, c0 * kC - 1).y : 0.0f;
  bool ok = true;
  // the copy after the last replayed update (reference: the running maximum before c0)
  if (c0 > 0)
    ok = state_copy<EPQ>(ms, tm, base, wq, hb, t, c0 - 1, 0, xfirst, Mp, Mc, lim);
  for (int c = c0; c < c1 && ok; ++c) {
    const int st = c % kNST;
    const int wi = c - c0;
    const float Mnn = c + 2 < c1 ? chunk_ref(scal, c + 2, N) : 0.0f;
    if (!mbar_wait_warp_lim(&ms->opd[st], (uint32_t)(c / kNST) & 1u, &ms->abort, lim)) {
      ok = false;
      break;
    }
    const float4 cf = lds128f(base + WLay::COEF + (st * kC + t) * 16);
    const uint32_t col_s = base + WLay::COL + st * kC * 8;
    if (!mbar_wait_warp_lim(&ms->a_full, (uint32_t)wi & 1u, &ms->abort, lim)) {
      ok = false;
      break;
    }
    tc_fence_after();
    // ---- S = [i <= t] (Q K^T) o W: 16-column pieces up to this warp's diagonal block, the
    //      load of the next piece in flight while one is formed.  Piece h (tokens 16 h ..
    //      16 h + 15, one K step of S V) is written packed to columns 16 h .. 16 h + 7, inside
    //      the fp32 columns that the same thread has just read: the quadrant's E warps share
    //      no column, so neither overwrites what the other still has to read ----
    {
      const int npiece = 2 * (wq + 1);
      // W 2^kr from the coefficients (which carry 2^kb, and b also 2^ks)
      const float sw = cf.w * pow2f(-state_exp(c));
      const float wa = cf.x * cf.w, wb = cf.y * sw * sinv, wg = cf.z * sw;
      const float2 a2 = make_float2(wa, wa), b2 = make_float2(wb, wb);
      const float2 g2 = make_float2(wg, wg);
      uint32_t ra[2][16];
      auto piece = [&](int h, const uint32_t (&rv)[16]) {
        uint32_t pw[8];
#pragma unroll
        for (int y = 0; y < 8; ++y) {
          const float4 cc = lds128f(col_s + (8 * h + y) * 16);  // tokens 16h+2y, +1: (e, s, e', s')
          const float2 w2 = __ffma2_rn(a2, make_float2(cc.x, cc.z),
                                       __ffma2_rn(b2, make_float2(cc.y, cc.w), g2));
          float2 val = __fmul2_rn(make_float2(__uint_as_float(rv[2 * y]),
                                              __uint_as_float(rv[2 * y + 1])), w2);
          const int i0 = 16 * h + 2 * y;
          if ((h >> 1) == wq) {  // diagonal block: keep i <= t only
            if (i0 > t) val.x = 0.0f;
            if (i0 + 1 > t) val.y = 0.0f;
          }
          pw[y] = pack_f16x2(val.x, val.y);
        }
        tmem_st8_nowait(tm + TM_A + 16 * h, pw);
      };
      // this warp's pieces: h = hb, hb + EPQ, ... (the quadrant's E warps alternate)
      tmem_ld16_nowait(tm + TM_A + 16 * hb, ra[0]);
#pragma unroll 1
      for (int h = hb; h < npiece; h += 2 * EPQ) {
        tmem_wait_ld();
        reg_fence(ra[0]);
        const bool two = h + EPQ < npiece;
        if (two) tmem_ld16_nowait(tm + TM_A + 16 * (h + EPQ), ra[1]);
        piece(h, ra[0]);
        if (two) {
          tmem_wait_ld();
          reg_fence(ra[1]);
          if (h + 2 * EPQ < npiece) tmem_ld16_nowait(tm + TM_A + 16 * (h + 2 * EPQ), ra[0]);
          piece(h + EPQ, ra[1]);
        }
      }
      uint32_t zw[8];
#pragma unroll
      for (int y = 0; y < 8; ++y) zw[y] = 0u;
#pragma unroll 1
      for (int h = npiece + hb; h < kC / 16; h += EPQ) tmem_st8_nowait(tm + TM_A + 16 * h, zw);
      tmem_wait_st();
    }
    tc_fence_before();
    __syncwarp();
    // (the testing hook withholds the first arrival of warp kEpWarp0: the S V product's wait
    // then runs out and the CTA abandons its work)
    if ((threadIdx.x & 31) == 0 && !(p.dbg_skip && wi == 0 && (threadIdx.x >> 5) == kEpWarp0))
      mbar_arrive(&ms->s_full);
    // ---- the state after this chunk -> B tile of the next one ----
    if (c <= c1 - 2) {
      ok = state_copy<EPQ>(ms, tm, base, wq, hb, t, c, c - cfirst, xfirst, Mc, Mn, lim);
      if (!ok) break;
    }
    // ---- o = X_SV + a X_F + b X_G + g X_H (16-column pieces) ----
    if (!mbar_wait_warp_lim(&ms->x_full, (uint32_t)wi & 1u, &ms->abort, lim)) {
      ok = false;
      break;
    }
    tc_fence_after();
    const bool has_state = c > 0;
    const float rinv = __frcp_rn(cf.w);  // S V carries the row's 2^kr
    // the B tile's F~ is referenced to the running maximum before the chunk, and scaled by 2^-kb
    const float xa = has_state ? cf.x * (expf(Mp - Mc) * pow2f(state_exp(c))) : 0.0f;
    // outputs of columns 16 pc .. 16 pc + 15: two TMEM round trips of two matrices each
    auto out_piece = [&](int pc, float (&o)[16]) {
      uint32_t r0[16], r1[16];
      tmem_ld16_nowait(tm + TM_SV + 16 * pc, r0);
      if (has_state) tmem_ld16_nowait(tm + TM_X + 16 * pc, r1);
      tmem_wait_ld();
      reg_fence(r0);
      const float2 ri2 = make_float2(rinv, rinv);
      auto f2 = [](const uint32_t (&r)[16], int j) {
        return make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
      };
      if (has_state) {
        reg_fence(r1);
        const float2 xa2 = make_float2(xa, xa);
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const float2 y = __ffma2_rn(xa2, f2(r1, j), __fmul2_rn(f2(r0, j), ri2));
          o[j] = y.x;
          o[j + 1] = y.y;
        }
        tmem_ld16_nowait(tm + TM_X + 64 + 16 * pc, r0);
        tmem_ld16_nowait(tm + TM_X + 128 + 16 * pc, r1);
        tmem_wait_ld();
        reg_fence(r0);
        reg_fence(r1);
        const float2 yb2 = make_float2(cf.y, cf.y), yg2 = make_float2(cf.z, cf.z);
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const float2 y = __ffma2_rn(yg2, f2(r1, j),
                                      __ffma2_rn(yb2, f2(r0, j), make_float2(o[j], o[j + 1])));
          o[j] = y.x;
          o[j + 1] = y.y;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const float2 y = __fmul2_rn(f2(r0, j), ri2);
          o[j] = y.x;
          o[j + 1] = y.y;
        }
      }
    };
    // the staging tile is free once the previous chunk's store has read it
    if (wi >= 1) {
      if (leader) {
        bulk_wait_group_read0();
        mbar_arrive(&ms->ob_free);
      }
      if (!mbar_wait_warp_lim(&ms->ob_free, (uint32_t)(wi - 1) & 1u, &ms->abort, lim)) {
        ok = false;
        break;
      }
    }
#pragma unroll 1
    for (int pc = hb * (4 / EPQ); pc < (hb + 1) * (4 / EPQ); ++pc) {
      float o[16];
      out_piece(pc, o);
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const float* o8 = o + 8 * x;
        sts128(base + WLay::OUTS + sw128_off(t, 2 * pc + x),
               make_uint4(pack_bf16x2(o8[0], o8[1]), pack_bf16x2(o8[2], o8[3]),
                          pack_bf16x2(o8[4], o8[5]), pack_bf16x2(o8[6], o8[7])));
      }
    }
    tc_fence_before();
    fence_proxy_async_smem();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
      mbar_arrive(&ms->x_free);
      mbar_arrive(&ms->ob_full);
    }
    if (leader) {
      // every output warp has written its rows: store the chunk (the staging tile is handed
      // back before the next chunk's rows are written, once the store has read it)
      if (!mbar_wait(&ms->ob_full, (uint32_t)wi & 1u, &ms->abort, lim)) {
        ok = false;
      } else {
        tma_store_3d(&p.to, base + WLay::OUTS, 0, c * kC, bh);
        bulk_commit_group();
      }
    }
    ok = __all_sync(0xffffffffu, ok);
    Mp = Mc;
    Mc = Mn;
    Mn = Mnn;
  }
  if (leader) bulk_wait_group0();
  if (!ok) {
    fail_wait(ms, a.status);
    return;
  }
  // ---- final state (prefill) by the CTA holding the sequence's last chunk ----
  const int nch = (N + kC - 1) / kC;
  if (a.final_state && c1 == nch && c1 > 0) {
    if (!mbar_wait_warp_lim(&ms->fin, 0, &ms->never, lim)) {
      fail_wait(ms, a.status);
      return;
    }
    tc_fence_after();
    float* rec = record_ptr(a.final_state, bh, kD);
    const int j = wq < 2 ? t : t - 64;
    const float gs = pow2f(s_exp(a, bh));  // G was carried with s 2^-ks
    constexpr int W = 32 / EPQ;
    static_assert(W == 16, "two E warps per quadrant");
#pragma unroll 1
    for (int q = 0; q < kStPieces; ++q) {
      const Piece pc = st_piece(wq, t, q);
      uint32_t v[W];
      tmem_ld16_nowait(tm + pc.col + W * hb, v);
      tmem_wait_ld();
      reg_fence(v);
      const int off = pc.rec == 0 ? rec_F(kD) : pc.rec == 1 ? rec_G(kD) : rec_H(kD);
#pragma unroll
      for (int y = 0; y < W; ++y)
        rec[off + (pc.a0 + W * hb + y) * kD + j] = __uint_as_float(v[y]) * (pc.rec == 1 ? gs : 1.0f);
    }
  }
}

// ============================================================================ kernel
__global__ void __launch_bounds__(kThreads, 1) walk_kernel(const __grid_constant__ WalkParams p) {
  constexpr int kEw = 4 * kEpq;  // E warps
  const FwdArgs& a = p.a;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (smem_u32(smem) & 1023u) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) report(a.status, kErrUnsupported);
    return;
  }
  WMisc* ms = reinterpret_cast<WMisc*>(smem + WLay::MISC);
  const int warp = threadIdx.x >> 5;
  const int bh = blockIdx.x / p.nseg, sg = blockIdx.x % p.nseg;
  const int c0 = p.seg_start[sg], c1 = p.seg_start[sg + 1];

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNST; ++i) {
      mbar_init(&ms->full[i], 1);
      mbar_init(&ms->empty[i], 1);
      mbar_init(&ms->opd[i], kOpWarps);
    }
    mbar_init(&ms->vsc_free, 1);
    mbar_init(&ms->a_full, 1);
    mbar_init(&ms->s_full, kEw);
    mbar_init(&ms->x_full, 1);
    mbar_init(&ms->x_free, kEw);
    mbar_init(&ms->u_done, 1);
    mbar_init(&ms->st_done, kEw);
    mbar_init(&ms->sb_free, 1);
    mbar_init(&ms->ob_free, 1);
    mbar_init(&ms->ob_full, kEw);
    mbar_init(&ms->fin, 1);
    ms->abort = 0;
    ms->never = 0;
  }
  if (a.rope && threadIdx.x < 32)  // rotary frequencies
    reinterpret_cast<float*>(smem + WLay::THETA)[threadIdx.x] = p.ang[threadIdx.x];
  if (warp == kMmaWarp) {
    tmem_alloc(&ms->tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // launched as a programmatic dependent of the scalar pass: every read of its output follows
  grid_dep_wait();

  if (warp < kOpWarps) {
    role_op(p, smem, ms, bh, c0, c1);
  } else if (warp < kMmaWarp) {
    role_e(p, smem, ms, bh, c0, c1);
  } else if (warp == kMmaWarp) {
    role_mma(p, smem, ms, c0, c1);
  } else if ((threadIdx.x & 31) == 0) {
    role_tma(p, smem, ms, bh, c0, c1);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    // every MMA has completed once `fin` fires (it is committed after the last one)
    if (!mbar_wait(&ms->fin, 0, &ms->never, 4000000000ll)) report(a.status, kErrTimeout);
    tc_fence_after();
    tmem_dealloc(ms->tmem, 512);
  }
}

// Rotary angles of the d = 64 walk: theta_a = base^(-2a/64) (a < 32), then for every chunk c
// the base angle c * 128 * theta_a reduced modulo 2 pi, both computed in fp64 and stored fp32.
__global__ void walk_angle_kernel(float* tab, int nch, double base) {
  const double two_pi = 6.283185307179586476925286766559;
  const int total = (nch + 1) * 32;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += gridDim.x * blockDim.x) {
    const int row = idx / 32, pa = idx % 32;
    const double theta = pow(base, -2.0 * (double)pa / (double)kD);
    if (row == 0) {
      tab[idx] = (float)theta;
    } else {
      const double ang = (double)(row - 1) * kC * theta;
      tab[idx] = (float)(ang - rint(ang * (1.0 / two_pi)) * two_pi);
    }
  }
}

std::atomic<long long> g_dbg_wait_limit{0};  // zeros_debug_walk settings (off by default)
std::atomic<int> g_dbg_skip{0};

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

// [B*H, N, 64] bf16 tensor viewed as 3-D (d fastest), boxes of {64, 128 tokens, 1 sequence},
// 128-byte swizzle.  Loads past N read zeros; stores past N are dropped.
bool make_map(CUtensorMap* m, const void* ptr, int N, int BH) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)N * (cuuint64_t)kD * 2};
  const cuuint32_t box[3] = {(cuuint32_t)kD, (cuuint32_t)kC, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count(int dev) {
  static std::atomic<int> cache[64];
  if (dev < 0 || dev >= 64) return 148;
  int v = cache[dev].load();
  if (v <= 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 148;
    cache[dev].store(v);
  }
  return v;
}

cudaError_t launch_walk(const FwdArgs& a, const float* ang, int nseg_max, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_set{0};  // bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)WLay::BYTES);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  WalkParams p;
  p.a = a;
  p.ang = ang;
  const long long lim = g_dbg_wait_limit.load();
  p.wait_limit = lim > 0 ? lim : 4294967296ll;
  p.dbg_skip = g_dbg_skip.load();
  const int BH = a.B * a.H;
  if (!make_map(&p.tq, a.q, a.N, BH) || !make_map(&p.tk, a.k, a.N, BH) ||
      !make_map(&p.tv, a.v, a.N, BH) || !make_map(&p.to, a.out, a.N, BH))
    return cudaErrorNotSupported;
  // segments per sequence: as many as the SMs allow (one CTA each), at most kMaxSeg and one
  // per chunk; segment j gets a share proportional to (1 - rho)^j, rho the cost of replaying
  // a chunk's state side relative to walking it (0.55 timed best at 64 sequences of 32 chunks,
  // between 0.4 and 0.85: the replay is bound by the operand warps, which still rotate and scale
  // every key), so that every CTA does about the same work
  const int nch = (a.N + kC - 1) / kC;
  const int nsm = sm_count(dev);
  int S = BH >= nsm ? 1 : nsm / BH;
  S = std::min(S, std::min(kMaxSeg, nseg_max));
  S = std::max(1, std::min(S, nch));
  constexpr double rho = 0.55;
  double wsum = 0.0, wj = 1.0;
  for (int j = 0; j < S; ++j, wj *= 1.0 - rho) wsum += wj;
  p.nseg = S;
  p.seg_start[0] = 0;
  double acc = 0.0;
  wj = 1.0;
  for (int j = 1; j <= S; ++j, wj *= 1.0 - rho) {
    acc += wj;
    int cj = (j == S) ? nch : (int)llround(nch * acc / wsum);
    cj = std::max(cj, p.seg_start[j - 1] + 1);       // every segment at least one chunk
    cj = std::min(cj, nch - (S - j));                 // and room for the ones after it
    p.seg_start[j] = cj;
  }
  for (int j = S + 1; j <= kMaxSeg; ++j) p.seg_start[j] = nch;
  const long long ctas = (long long)BH * S;
  if (ctas > 0x7fffffffll) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = WLay::BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, walk_kernel, p);
  count_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool walk_supported(int d, int dtype, int causal) { return d == kD && dtype == 0 && causal == 1; }

void set_walk_debug(long long wait_limit_cycles, int skip_one_arrive) {
  g_dbg_wait_limit.store(wait_limit_cycles);
  g_dbg_skip.store(skip_one_arrive ? 1 : 0);
}

size_t walk_angle_floats(int N) { return (size_t)((N + kC - 1) / kC + 1) * 32; }

cudaError_t launch_walk_angles(float* tab, int N, double base, cudaStream_t stream) {
  const int nch = (N + kC - 1) / kC;
  const int total = (nch + 1) * 32;
  const int blocks = std::min(1024, (total + 255) / 256);
  walk_angle_kernel<<<std::max(blocks, 1), 256, 0, stream>>>(tab, nch, base);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_fwd_walk(const FwdArgs& a, const float* ang, int nseg_max,
                            cudaStream_t stream) {
  // (the fused output LayerNorm runs on the chunked kernel of zs_chunk.cu)
  if (!a.scal || !a.smax || (a.rope && !ang) || a.ln) return cudaErrorInvalidValue;
  return launch_walk(a, ang, nseg_max, stream);
}

}  // namespace zs
