// Per-token scalars of the causal ZeroS layer for whole sequences, ahead of the chunked
// tensor-core forward.
//
// Method: Paper-Notes "ZeroS: Zero-Sum Linear Attention for Efficient Transformers", method
// details: the deviation logits s_i = -(1/sqrt d) u_i ubar_i^T with the prior-smoothed mean
// ubar_i, and the prefix sums E_t = sum e^{s_i}, P_t = sum s_i of the "linear-time prefix scan".
// They are evaluated in the blocked fp32 order of zs_common.cuh (32-token blocks, every running
// quantity a carry plus a block-local value), which makes them bit-identical to the decode step
// and to the token-sequential forward.
//
// The order has two sequential chains per sequence, one add per block: the column sums of u
// (the carry C) and the scalar carries (mC, EC, CP).  Everything else is local to a block.  So a
// sequence is processed by one cluster of kScCN CTAs, in segments of kScCN x kScW x BW blocks
// (BW = 2 blocks per warp at d = 64, 1 at d = 128); each warp owns BW consecutive blocks of a
// segment:
//   A. each block's local column sums L (fp32, token order), stored into the shared memory of
//      every CTA of the cluster (remote stores, then a cluster barrier);
//   B. warp 0 of every CTA walks the segment's blocks in order through its own copy and records
//      the column carry at the start of its own blocks;
//   C. each warp forms its tokens' logits (same lane/tree order as the decode step), the
//      block-local running max, scaled exp-sum and logit sum, and stores the block's end values
//      into every CTA of the cluster;
//   D. the end values are folded in block order (the same fold as the decode step), recording
//      the scalar carries at the start of every block: the maximum chain first (a prefix
//      maximum across the lanes of warp 0), then the exponentials of every block at once, then
//      the multiply-add and add chains (warps 0 and 1), so that only one operation per block
//      is sequential;
//   E. each token combines its block's carries with its local values: (s, m, Et, P).
// Output: float4 (s, m, Et, P) per token, [B*H, N] (16 bytes per token); optionally the debug
// scalars and the scalar part of the recurrent state after the last token (C, L, mu and the
// record head), in the layout of the decode state.
#include <math.h>

#include <atomic>

#include "zs_common.cuh"
#include "zs_internal.h"
#include "zs_sm100.cuh"

namespace zs {
namespace {

using namespace sm100;

constexpr int kScCN = kScalarCtas;  // CTAs per sequence (one cluster)
constexpr int kScW = 8;   // warps per CTA

// Blocks per warp and per segment: two at d = 64 (a 4096-token sequence is one segment).
template <int D>
struct ScShape {
  static constexpr int BW = (D == 64) ? 2 : 1;      // blocks per warp
  static constexpr int CB = kScW * BW;              // blocks per CTA
  static constexpr int SEG = kScCN * CB;            // blocks per segment
};

struct BlockCarry {
  float mC, EC, CP;
};

// Fold a block's end values (LP, ml, El) into the carries (the block-end step of the contract).
__device__ __forceinline__ void fold_block(BlockCarry& k, float LP, float ml, float El) {
  const float P = __fadd_rn(k.CP, LP);
  const float m = fmaxf(k.mC, ml);
  const float Et = __fmaf_rn(k.EC, expf(__fsub_rn(k.mC, m)), __fmul_rn(El, expf(__fsub_rn(ml, m))));
  k.CP = P;
  k.mC = m;
  k.EC = Et;
}

template <int D>
struct ScSmem {
  using SH = ScShape<D>;
  float lend[SH::SEG][D];    // local column sums of every block of the segment (all CTAs write)
  float4 bend[SH::SEG];      // end values (LP, ml, El, -) of every block (all CTAs write)
  float cw[SH::CB][D];       // column carry at the start of each of this CTA's blocks
  // per block of the segment: the fold's two exponential terms fx, fy and its LP (fz), and the
  // carries (mC, EC, CP) at the block's start
  __align__(16) float fx[SH::SEG];
  __align__(16) float fy[SH::SEG];
  __align__(16) float fz[SH::SEG];
  __align__(16) float cm[SH::SEG];
  __align__(16) float cEC[SH::SEG];
  __align__(16) float cCP[SH::SEG];
  float kseg[3];             // carries (mC, EC, CP) at the current segment's start
  float4 chain[kScW][32];    // per warp: (s, e^{ml_{j-1} - ml_j}, e^{s - ml_j}, -) of token j
  float4 loc[SH::CB][32];    // per token of this CTA's blocks: (s, ml, El, LP), block-local
  int smax_bits;             // largest |s| of this CTA's tokens (bits of a non-negative float)
};

// Lane's R = D / 32 columns of token row j (bf16 pairs as float2), zero past the sequence.
template <int D>
__device__ __forceinline__ void load_row(const __nv_bfloat16* urow, bool valid,
                                         float2 (&o)[D / 64]) {
  constexpr int R = D / 32;
  if (R == 2) {
    const uint32_t wv = valid ? __ldg(reinterpret_cast<const unsigned int*>(urow)) : 0u;
    unpack_bf16x2(wv, o[0].x, o[0].y);
  } else {
    const uint2 wv = valid ? __ldg(reinterpret_cast<const uint2*>(urow)) : make_uint2(0u, 0u);
    unpack_bf16x2(wv.x, o[0].x, o[0].y);
    unpack_bf16x2(wv.y, o[D / 64 - 1].x, o[D / 64 - 1].y);
  }
}

template <int D>
__global__ void __cluster_dims__(kScCN, 1, 1) __launch_bounds__(kScW * 32, D == 64 ? 4 : 2)
    scal_kernel(const FwdArgs a, float4* __restrict__ scal) {
  constexpr int R = D / 32;  // columns per lane: 2 or 4
  constexpr int RP = R / 2;  // column pairs per lane
  using SH = ScShape<D>;
  constexpr int BW = SH::BW, CB = SH::CB, SEG = SH::SEG;
  extern __shared__ __align__(16) uint8_t sc_raw[];
  ScSmem<D>& sm = *reinterpret_cast<ScSmem<D>*>(sc_raw);
  const uint32_t rank = cluster_rank();
  const int bh = blockIdx.x / kScCN, h = bh % a.H;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;
  const size_t row0 = (size_t)bh * N;
  const int nb = (N + 31) / 32;
  const int nseg = (nb + SEG - 1) / SEG;
  const float etau = expf(a.tau[h]);
  const float sqrtd = __fsqrt_rn((float)D);
  const float2 etau2 = make_float2(etau, etau);
  const __nv_bfloat16* ucol = static_cast<const __nv_bfloat16*>(a.u) + row0 * D + R * lane;
  float2 mu2[RP];
#pragma unroll
  for (int x = 0; x < RP; ++x)
    mu2[x] = make_float2(a.mu[(size_t)h * D + R * lane + 2 * x],
                         a.mu[(size_t)h * D + R * lane + 2 * x + 1]);
  // carries at the current segment's start (kept by warp 0 of every CTA)
  float2 Cseg[RP];
#pragma unroll
  for (int x = 0; x < RP; ++x) Cseg[x] = make_float2(0.0f, 0.0f);
  float amax = 0.0f;  // largest |s| of this thread's tokens
  if (threadIdx.x == 0) {
    sm.smax_bits = 0;
    sm.kseg[0] = -INFINITY;  // scalar carries (mC, EC, CP) at the segment's start
    sm.kseg[1] = 0.0f;
    sm.kseg[2] = 0.0f;
  }

  for (int sg = 0; sg < nseg; ++sg) {
    // this warp's blocks: segment blocks gi0 .. gi0 + BW - 1
    const int gi0 = (int)rank * CB + w * BW;
    int b0[BW], nvalid[BW];
#pragma unroll
    for (int bb = 0; bb < BW; ++bb) {
      b0[bb] = (sg * SEG + gi0 + bb) * 32;
      nvalid[bb] = max(0, min(32, N - b0[bb]));
    }
    // ---- A: local column sums of each block (token order), to every CTA of the cluster ----
#pragma unroll 1
    for (int bb = 0; bb < BW; ++bb) {
      float2 L[RP];
#pragma unroll
      for (int x = 0; x < RP; ++x) L[x] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float2 uj[RP];
        load_row<D>(ucol + (size_t)(b0[bb] + j) * D, j < nvalid[bb], uj);
#pragma unroll
        for (int x = 0; x < RP; ++x) L[x] = __fadd2_rn(L[x], uj[x]);
      }
      const uint32_t dst = smem_u32(&sm.lend[gi0 + bb][R * lane]);
#pragma unroll
      for (uint32_t cr = 0; cr < (uint32_t)kScCN; ++cr) {
        if (RP == 1) st_cluster_f32x2(mapa(dst, cr), L[0].x, L[0].y);
        else st_cluster_f32x4(mapa(dst, cr), make_float4(L[0].x, L[0].y, L[RP - 1].x, L[RP - 1].y));
      }
    }
    cluster_sync_all();
    // ---- B: column carry at the start of every block of the segment (block order); the sums
    //      of the next 8 blocks are loaded while the chain runs over the current 8 ----
    if (w == 0) {
      constexpr int G = 8;
      static_assert(SEG % (2 * G) == 0, "whole pairs of groups per segment");
      float2 Cc[RP];
#pragma unroll
      for (int x = 0; x < RP; ++x) Cc[x] = Cseg[x];
      float2 la[G][RP], lb[G][RP];
      auto load_group = [&](float2 (&le)[G][RP], int g0) {
#pragma unroll
        for (int i = 0; i < G; ++i)
#pragma unroll
          for (int x = 0; x < RP; ++x)
            le[i][x] = *reinterpret_cast<const float2*>(&sm.lend[g0 + i][R * lane + 2 * x]);
      };
      auto chain_group = [&](const float2 (&le)[G][RP], int g0) {
        const bool own = g0 / CB == (int)rank;  // a group of 8 lies within one CTA's blocks
#pragma unroll
        for (int i = 0; i < G; ++i) {
          if (own) {
#pragma unroll
            for (int x = 0; x < RP; ++x)
              *reinterpret_cast<float2*>(&sm.cw[(g0 + i) % CB][R * lane + 2 * x]) = Cc[x];
          }
#pragma unroll
          for (int x = 0; x < RP; ++x) Cc[x] = __fadd2_rn(Cc[x], le[i][x]);
        }
      };
      load_group(la, 0);
#pragma unroll 1
      for (int g0 = 0; g0 < SEG; g0 += 2 * G) {
        load_group(lb, g0 + G);
        chain_group(la, g0);
        if (g0 + 2 * G < SEG) load_group(la, g0 + 2 * G);
        chain_group(lb, g0 + G);
      }
#pragma unroll
      for (int x = 0; x < RP; ++x) Cseg[x] = Cc[x];
    }
    __syncthreads();
    // ---- C: logits (two tokens per f32x2 step) and the block-local chains, block by block ----
#pragma unroll 1
    for (int bb = 0; bb < BW; ++bb) {
      float2 Lc[RP], Cw[RP];
#pragma unroll
      for (int x = 0; x < RP; ++x) {
        Cw[x] = *reinterpret_cast<const float2*>(&sm.cw[w * BW + bb][R * lane + 2 * x]);
        Lc[x] = make_float2(0.0f, 0.0f);
      }
      float pp[32];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        // at most 16 rows of loads in flight (they are L2 hits): bounds the live registers
        if (j == 16) asm volatile("" ::: "memory");
        float2 u0[RP], u1[RP];
        load_row<D>(ucol + (size_t)(b0[bb] + j) * D, j < nvalid[bb], u0);
        load_row<D>(ucol + (size_t)(b0[bb] + j + 1) * D, j + 1 < nvalid[bb], u1);
        float2 n0[RP], n1[RP];
#pragma unroll
        for (int x = 0; x < RP; ++x) {
          Lc[x] = __fadd2_rn(Lc[x], u0[x]);
          n0[x] = __ffma2_rn(etau2, mu2[x], __fadd2_rn(Cw[x], Lc[x]));
          Lc[x] = __fadd2_rn(Lc[x], u1[x]);
          n1[x] = __ffma2_rn(etau2, mu2[x], __fadd2_rn(Cw[x], Lc[x]));
        }
        // p = u[R l] n[R l], then fma over the lane's remaining columns, for tokens j and j + 1
        float2 p = __fmul2_rn(make_float2(u0[0].x, u1[0].x), make_float2(n0[0].x, n1[0].x));
#pragma unroll
        for (int col = 1; col < R; ++col) {
          const int x = col >> 1;
          const float a0 = (col & 1) ? u0[x].y : u0[x].x, a1 = (col & 1) ? u1[x].y : u1[x].x;
          const float m0 = (col & 1) ? n0[x].y : n0[x].x, m1 = (col & 1) ? n1[x].y : n1[x].x;
          p = __ffma2_rn(make_float2(a0, a1), make_float2(m0, m1), p);
        }
        pp[j] = p.x;
        pp[j + 1] = p.y;
      }
      // transpose-reduce: the butterfly tree of the contract for 32 tokens at once; afterwards
      // lane j holds the full dot of token b0 + j
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
      const int i = b0[bb] + lane;
      const bool valid = lane < nvalid[bb];
      const float den = __fmul_rn(__fadd_rn(etau, (float)(i + 1)), sqrtd);
      const float s = -__fdiv_rn(pp[0], den);
      if (valid && !isfinite(s)) report(a.status, kErrRange);
      if (valid) amax = fmaxf(amax, fabsf(s));
      float ml = valid ? s : -INFINITY;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float x = __shfl_up_sync(0xffffffffu, ml, o);
        if (lane >= o) ml = fmaxf(ml, x);
      }
      float mlp = __shfl_up_sync(0xffffffffu, ml, 1);
      if (lane == 0) mlp = -INFINITY;
      __syncwarp();
      sm.chain[w][lane] = make_float4(s, expf(__fsub_rn(mlp, ml)), expf(__fsub_rn(s, ml)), 0.0f);
      __syncwarp();
      float LP = 0.0f, El = 0.0f;
      const int kend = min(nvalid[bb], lane + 1);  // this lane accumulates tokens 0 .. lane
#pragma unroll 8
      for (int k = 0; k < 32; ++k) {
        const float4 e = sm.chain[w][k];
        if (k < kend) {
          LP = __fadd_rn(LP, e.x);
          El = __fmaf_rn(El, e.y, e.z);
        }
      }
      if (lane == 31) {  // block end values (tokens 0 .. nvalid - 1) to every CTA of the cluster
        const uint32_t dst = smem_u32(&sm.bend[gi0 + bb]);
#pragma unroll
        for (uint32_t cr = 0; cr < (uint32_t)kScCN; ++cr)
          st_cluster_f32x4(mapa(dst, cr), make_float4(LP, ml, El, 0.0f));
      }
      sm.loc[w * BW + bb][lane] = make_float4(s, ml, El, LP);
    }
    cluster_sync_all();
    // ---- D: scalar carries at the start of every block of the segment (block order).  The
    //      maximum chain is an exact prefix maximum (lane l of warp 0 takes blocks Q l ..
    //      Q l + Q - 1; a maximum is exact, so any grouping gives the chain's values), and the
    //      exponentials of every block are formed at once.  The two remaining chains then run
    //      in block order on two warps (two schedulers), each one FMA per block with its
    //      operands read four blocks at a time ahead of the chain: EC = fma(EC, x, y) on warp 0,
    //      CP + z on warp 1 ----
    if (w == 0) {
      constexpr int Q = SEG / 32;
      float pre[Q];
#pragma unroll
      for (int i = 0; i < Q; ++i) {
        const float x = sm.bend[Q * lane + i].y;
        pre[i] = i == 0 ? x : fmaxf(pre[i - 1], x);
      }
      float incl = pre[Q - 1];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl = fmaxf(incl, y);
      }
      const float excl = __shfl_up_sync(0xffffffffu, incl, 1);
      const float mC = sm.kseg[0];
      const float base = lane == 0 ? mC : fmaxf(mC, excl);
#pragma unroll
      for (int i = 0; i < Q; ++i) {
        const int gb = Q * lane + i;
        const float mb = i == 0 ? base : fmaxf(base, pre[i - 1]);
        const float ma = fmaxf(base, pre[i]);
        const float4 be = sm.bend[gb];
        sm.fx[gb] = expf(__fsub_rn(mb, ma));
        sm.fy[gb] = __fmul_rn(be.z, expf(__fsub_rn(be.y, ma)));
        sm.fz[gb] = be.x;
        sm.cm[gb] = mb;
      }
      const float mrun = __shfl_sync(0xffffffffu, fmaxf(base, pre[Q - 1]), 31);
      __syncwarp();
      if (lane == 0) sm.kseg[0] = mrun;
    }
    __syncthreads();
    if (w < 2) {
      // every lane alike: broadcast loads, stores of one value
      float acc = sm.kseg[1 + w];
      const float* mul = sm.fx;
      const float* add = w == 0 ? sm.fy : sm.fz;
      float* out = w == 0 ? sm.cEC : sm.cCP;
#pragma unroll
      for (int g = 0; g < SEG; g += 4) {
        const float4 a4 = *reinterpret_cast<const float4*>(add + g);
        float4 c;
        if (w == 0) {
          const float4 m4 = *reinterpret_cast<const float4*>(mul + g);
          c.x = acc; acc = __fmaf_rn(acc, m4.x, a4.x);
          c.y = acc; acc = __fmaf_rn(acc, m4.y, a4.y);
          c.z = acc; acc = __fmaf_rn(acc, m4.z, a4.z);
          c.w = acc; acc = __fmaf_rn(acc, m4.w, a4.w);
        } else {
          c.x = acc; acc = __fadd_rn(acc, a4.x);
          c.y = acc; acc = __fadd_rn(acc, a4.y);
          c.z = acc; acc = __fadd_rn(acc, a4.z);
          c.w = acc; acc = __fadd_rn(acc, a4.w);
        }
        *reinterpret_cast<float4*>(out + g) = c;
      }
      __syncwarp();
      if (lane == 0) sm.kseg[1 + w] = acc;
    }
    __syncthreads();
    // ---- E: each token's scalars ----
#pragma unroll 1
    for (int bb = 0; bb < BW; ++bb) {
      // the block's carries (mC, EC, CP) at its start
      const float4 kc = make_float4(sm.cm[gi0 + bb], sm.cEC[gi0 + bb], sm.cCP[gi0 + bb], 0.0f);
      const float4 lv = sm.loc[w * BW + bb][lane];
      const float s = lv.x, ml = lv.y, El = lv.z, LP = lv.w;
      const int i = b0[bb] + lane;
      const float P = __fadd_rn(kc.z, LP);
      const float m = fmaxf(kc.x, ml);
      const float Et = __fmaf_rn(kc.y, expf(__fsub_rn(kc.x, m)), __fmul_rn(El, expf(__fsub_rn(ml, m))));
      if (lane < nvalid[bb]) {
        scal[row0 + i] = make_float4(s, m, Et, P);
        if (a.dbg_s) a.dbg_s[row0 + i] = s;
        if (a.dbg_E) a.dbg_E[row0 + i] = Et;
        if (a.dbg_P) a.dbg_P[row0 + i] = P;
        if (a.dbg_m) a.dbg_m[row0 + i] = m;
      }
      // recurrent state after the last token (prefill), by the warp owning that token
      if (a.final_state && nvalid[bb] > 0 && b0[bb] + nvalid[bb] == N) {
        float* rec = record_ptr(a.final_state, bh, D);
        const bool closed = nvalid[bb] == 32;  // a complete block: folded as the decode step does
        const float LPe = __shfl_sync(0xffffffffu, LP, 31);
        const float mle = __shfl_sync(0xffffffffu, ml, 31);
        const float Ele = __shfl_sync(0xffffffffu, El, 31);
        BlockCarry kf{kc.x, kc.y, kc.z};
        if (closed) fold_block(kf, LPe, mle, Ele);
#pragma unroll
        for (int x = 0; x < RP; ++x) {
#pragma unroll
          for (int y = 0; y < 2; ++y) {
            const int col = R * lane + 2 * x + y;
            const float cw = sm.cw[w * BW + bb][col], le = sm.lend[gi0 + bb][col];
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
  // the CTA's largest |s| (non-negative floats order like their bit patterns)
  if (a.smax) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) atomicMax(&sm.smax_bits, __float_as_int(amax));
    __syncthreads();
    if (threadIdx.x == 0) a.smax[(size_t)bh * kScCN + rank] = __int_as_float(sm.smax_bits);
  }
  // (no remote access follows the last cluster barrier)
  grid_dep_launch();  // the forward kernel may be scheduled; it waits for this grid's completion
}


template <int D>
cudaError_t launch_scal_d(const FwdArgs& a, float4* scal, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_set{0};  // bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(scal_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(ScSmem<D>));
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  const long long ctas = (long long)a.B * a.H * kScCN;
  if (ctas > 0x7fffffffll) return cudaErrorInvalidValue;
  scal_kernel<D><<<dim3((unsigned)ctas), dim3(kScW * 32), sizeof(ScSmem<D>), stream>>>(a, scal);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_scalars(const FwdArgs& a, float4* scal, cudaStream_t stream) {
  if (a.d == 64) return launch_scal_d<64>(a, scal, stream);
  if (a.d == 128) return launch_scal_d<128>(a, scal, stream);
  return cudaErrorInvalidValue;
}

}  // namespace zs
