// Token-sequential CUDA-core forward of the ZeroS layer (causal and encoder modes), plus the
// small utility kernels (state init / header, rotary tables).
//
// Method: Paper-Notes "ZeroS: Zero-Sum Linear Attention for Efficient Transformers", method
// details, "linear-time prefix scan": the five prefix states E, P, F, G, H are updated once per
// token and read out as o_t = q_hat_t (alpha_t F_t + beta_t G_t + gamma_t H_t).  This kernel
// does exactly that, one token after the other, with the fp32 states in registers.  It is the
// fp32-input path and the reference CUDA path against which the chunked tensor-core kernel is
// checked; it is not the bf16 fast path.
//
// Grid: one CTA per (b, h, 32-wide slice of the value columns); 256 threads = 8 warps.  Warp w,
// lane l own state rows a = w + 8 r and value column j0 + l of F~ (= F e^{-m}), G and H.
// Warp 0 also runs the canonical token update of zs_common.cuh (logit, m, Et, P); warps 1..3
// normalise / rotate q_t and k_t and stage v_t in shared memory.
#include <math.h>


#include "zs_common.cuh"
#include "zs_internal.h"
#include "zs_sm100.cuh"

namespace zs {
namespace {

using namespace sm100;

constexpr int kThreads = 256;

struct TokenCoefs {
  float s, f, g, alpha, beta, gamma;
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) fwd_simt_kernel(FwdArgs a) {
  constexpr int R = D / 32;  // columns per lane in a warp-owned row
  constexpr int RA = D / 8;  // state rows per thread
  const int bh = blockIdx.x;
  const int h = bh % a.H;
  const int j0 = blockIdx.y * 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;
  const size_t row0 = (size_t)bh * N;
  const T* __restrict__ q = static_cast<const T*>(a.q) + row0 * D;
  const T* __restrict__ k = static_cast<const T*>(a.k) + row0 * D;
  const T* __restrict__ v = static_cast<const T*>(a.v) + row0 * D;
  const T* __restrict__ u = static_cast<const T*>(a.u) + row0 * D;
  T* __restrict__ out = static_cast<T*>(a.out) + row0 * D;
  const float* __restrict__ g1 = a.g1 + row0;
  const float* __restrict__ gh = a.gh + row0;

  __shared__ float qs[D], ks[D], vs[32];
  __shared__ float red[8][32];
  __shared__ TokenCoefs tc;

  // Output LayerNorm over the head's d columns.  The d/32 value slices of a head form one
  // cluster (launched so when ln is set and d > 32).  Warp 7 writes the outputs: for token t it
  // publishes (mean, M2) of its 32 columns to the other slices, then normalises token t - 1,
  // whose statistics have had a token's time to arrive.
  constexpr int NSL = D / 32;
  __shared__ float2 lnx[2][NSL];                 // [token parity][slice]
  __shared__ __align__(8) uint64_t ln_full[2];   // one arrival per other slice
  __shared__ int ln_abort;
  const bool clustered = a.ln && NSL > 1;
  const int me = blockIdx.y;
  if (clustered) {
    if (threadIdx.x == 0) {
      mbar_init(&ln_full[0], NSL - 1);
      mbar_init(&ln_full[1], NSL - 1);
      ln_abort = 0;
      fence_mbarrier_init_cluster();
    }
    cluster_sync_all();
  }
  float ln_w = 1.0f, ln_b = 0.0f;
  if (a.ln && warp == 7) {
    if (a.ln_w) ln_w = a.ln_w[(size_t)h * D + j0 + lane];
    if (a.ln_b) ln_b = a.ln_b[(size_t)h * D + j0 + lane];
  }
  float prev_o = 0.0f, prev_mean = 0.0f, prev_m2 = 0.0f;
  bool ln_ok = true;
  // warp 7: normalise and store token tt (its output, mean and M2 held in prev_*)
  auto ln_finish = [&](int tt) {
    float n = 32.0f, mean = prev_mean, m2 = prev_m2;
    if (clustered && ln_ok) {
      ln_ok = mbar_wait_cl_warp(&ln_full[tt & 1], (uint32_t)(tt >> 1) & 1u, &ln_abort);
      if (!ln_ok) report(a.status, kErrTimeout);
#pragma unroll
      for (int r = 1; r < NSL; ++r) {
        const float2 o = lnx[tt & 1][(me + r) % NSL];
        moments_merge(n, mean, m2, 32.0f, o.x, o.y);
      }
    }
    const float rstd = rsqrtf(m2 * (1.0f / D) + a.ln_eps);
    st(out, (size_t)tt * D + j0 + lane, __fmaf_rn((prev_o - mean) * rstd, ln_w, ln_b));
  };
  // warp 7: output o of token tt (lane = column j0 + lane)
  auto emit = [&](int tt, float o) {
    if (!a.ln) {
      st(out, (size_t)tt * D + j0 + lane, o);
      return;
    }
    const float mean = warp_sum32(o) * (1.0f / 32.0f);
    const float dv = o - mean;
    const float m2 = warp_sum32(dv * dv);
    if (tt >= 1) ln_finish(tt - 1);
    if (clustered && ln_ok && lane == 0) {
#pragma unroll
      for (int r = 1; r < NSL; ++r) {
        const uint32_t peer = (uint32_t)((me + r) % NSL);
        st_cluster_f32x2(mapa(smem_u32(&lnx[tt & 1][me]), peer), mean, m2);
        mbar_arrive_remote(mapa(smem_u32(&ln_full[tt & 1]), peer));
      }
    }
    prev_o = o;
    prev_mean = mean;
    prev_m2 = m2;
  };

  float F[RA], G[RA], Hs[RA];
#pragma unroll
  for (int r = 0; r < RA; ++r) F[r] = G[r] = Hs[r] = 0.0f;

  // Warp-0 scalar state (canonical order of zs_common.cuh; lane owns columns R lane + r).
  float C[R], L[R], mu[R], nfix[R];
  Scalars sc = scalars_init();
  float m_run = -INFINITY, Et_run = 0.0f, P_run = 0.0f;  // encoder chains
  const float etau = expf(a.tau[h]);
  float den_fix = 0.0f;
  if (warp == 0) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      C[r] = 0.0f;
      L[r] = 0.0f;
      mu[r] = a.mu[(size_t)h * D + R * lane + r];
    }
    if (!a.causal) {
      // Encoder: full-sequence prior mean, numerator e^tau mu + sum_j u_j.
      float Su[R];
#pragma unroll
      for (int r = 0; r < R; ++r) Su[r] = 0.0f;
      for (int i = 0; i < N; ++i) {
#pragma unroll
        for (int r = 0; r < R; ++r) Su[r] = __fadd_rn(Su[r], ld(u, (size_t)i * D + R * lane + r));
      }
#pragma unroll
      for (int r = 0; r < R; ++r) nfix[r] = __fmaf_rn(etau, mu[r], Su[r]);
      den_fix = __fmul_rn(__fadd_rn(etau, (float)N), __fsqrt_rn((float)D));
      // the full-sequence scalars first: m_N, Et_N = E_N e^{-m_N}, P_N
      for (int i = 0; i < N; ++i) {
        float uu[R];
#pragma unroll
        for (int r = 0; r < R; ++r) uu[r] = ld(u, (size_t)i * D + R * lane + r);
        const float si = fixed_logit<R>(uu, nfix, den_fix);
        const float m_new = fmaxf(m_run, si);
        Et_run = __fmaf_rn(Et_run, expf(__fsub_rn(m_run, m_new)), expf(__fsub_rn(si, m_new)));
        P_run = __fadd_rn(P_run, si);
        m_run = m_new;
      }
    }
  }
  // Encoder sums, centred: with t = N for every query the weight is
  //   w_i = (sig1 - sigh) / N (s_i - P_N / N) + sigh (e^{s_i - m} - Et_N / N) / Et_N,
  // so F and G are accumulated with the centred factors (e^{s_i - m_N} - Et_N / N) and
  // (s_i - P_N / N).  The readout then adds two sums that do not cancel each other, instead of
  // three full sums whose large parts cancel (which costs fp32 digits in proportion).
  const float ebar = warp == 0 && !a.causal ? __fdiv_rn(Et_run, (float)N) : 0.0f;
  const float sbar = warp == 0 && !a.causal ? __fdiv_rn(P_run, (float)N) : 0.0f;

  auto load_unit_row = [&](const T* src, int t, float* dst) {
    float x[R];
    float2 cs[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      x[r] = ld(src, (size_t)t * D + lane + 32 * r);
      cs[r] = make_float2(1.0f, 0.0f);
    }
    if (a.rope) {
      const float2* tab = a.rope_table + (size_t)t * (D / 2);
      if (R == 1) {
        cs[0] = tab[pair_index<R>(lane, 0)];
      } else {
#pragma unroll
        for (int r = 0; r < R / 2; ++r) cs[r] = tab[pair_index<R>(lane, r)];
      }
    }
    unit_rotate<R>(x, a.rope != 0, cs);
#pragma unroll
    for (int r = 0; r < R; ++r) dst[lane + 32 * r] = x[r];
  };

  // ---- pass over the tokens: state update (+ readout in causal mode) ----
  for (int t = 0; t < N; ++t) {
    if (warp == 0) {
      float uu[R];
#pragma unroll
      for (int r = 0; r < R; ++r) uu[r] = ld(u, (size_t)t * D + R * lane + r);
      float f, g, s, Et, P, m, s_raw;
      if (a.causal) {
        const TokenOut o = token_update<R>(uu, C, L, mu, etau, t + 1, sc);
        s = o.s;
        s_raw = s;
        Et = o.Et;
        P = o.P;
        m = o.m;
        f = expf(__fsub_rn(o.m_prev, m));
        g = expf(__fsub_rn(s, m));
      } else {
        s_raw = fixed_logit<R>(uu, nfix, den_fix);  // as in the pre-pass
        s = __fsub_rn(s_raw, sbar);
        f = 1.0f;
        g = __fsub_rn(expf(__fsub_rn(s_raw, m_run)), ebar);
        Et = Et_run;
        P = P_run;
        m = m_run;
      }
      if (lane == 0) {
        if (!isfinite(s_raw)) report(a.status, kErrRange);
        tc.s = s;
        tc.f = f;
        tc.g = g;
        if (a.causal) {
          const float sig1 = sigmoid(g1[t]), sigh = sigmoid(gh[t]);
          const float rt = __fdiv_rn(1.0f, (float)(t + 1));
          const float beta = __fmul_rn(__fsub_rn(sig1, sigh), rt);
          tc.alpha = __fdiv_rn(sigh, Et);
          tc.beta = beta;
          tc.gamma = -__fadd_rn(__fmul_rn(__fmul_rn(beta, P), rt), __fmul_rn(sigh, rt));
          // optional zero-order term of a first layer: every weight gains sig0 / t
          if (a.g0) tc.gamma = __fadd_rn(tc.gamma, __fmul_rn(sigmoid(a.g0[row0 + t]), rt));
          if (blockIdx.y == 0) {
            if (a.dbg_s) a.dbg_s[row0 + t] = s;
            if (a.dbg_E) a.dbg_E[row0 + t] = Et;
            if (a.dbg_P) a.dbg_P[row0 + t] = P;
            if (a.dbg_m) a.dbg_m[row0 + t] = m;
          }
        } else if (blockIdx.y == 0 && a.dbg_s) {
          a.dbg_s[row0 + t] = s_raw;
        }
      }
    } else if (warp == 1) {
      if (a.causal) load_unit_row(q, t, qs);
    } else if (warp == 2) {
      load_unit_row(k, t, ks);
    } else if (warp == 3) {
      vs[lane] = ld(v, (size_t)t * D + j0 + lane);
    }
    __syncthreads();
    const float s = tc.s, f = tc.f, g = tc.g;
    const float vj = vs[lane];
    float acc = 0.0f;
#pragma unroll
    for (int r = 0; r < RA; ++r) {
      const int ai = warp + 8 * r;
      const float kv = __fmul_rn(ks[ai], vj);
      F[r] = __fmaf_rn(F[r], f, __fmul_rn(g, kv));
      G[r] = __fmaf_rn(s, kv, G[r]);
      Hs[r] = __fadd_rn(Hs[r], kv);
      if (a.causal) {
        const float comb = __fmaf_rn(tc.alpha, F[r], __fmaf_rn(tc.beta, G[r], __fmul_rn(tc.gamma, Hs[r])));
        acc = __fmaf_rn(qs[ai], comb, acc);
      }
    }
    if (a.causal) red[warp][lane] = acc;
    __syncthreads();
    if (a.causal && warp == 7) {
      float o = red[0][lane];
#pragma unroll
      for (int w = 1; w < 8; ++w) o = __fadd_rn(o, red[w][lane]);
      emit(t, o);
    }
  }
  if (a.causal && a.ln && warp == 7 && N > 0) ln_finish(N - 1);

  if (a.causal) {
    // ---- optional final state (prefill for recurrent decoding) ----
    if (a.final_state) {
      float* rec = record_ptr(a.final_state, bh, D);
#pragma unroll
      for (int r = 0; r < RA; ++r) {
        const int ai = warp + 8 * r;
        rec[rec_F(D) + ai * D + j0 + lane] = F[r];
        rec[rec_G(D) + ai * D + j0 + lane] = G[r];
        rec[rec_H(D) + ai * D + j0 + lane] = Hs[r];
      }
      if (blockIdx.y == 0 && warp == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          rec[rec_C(D) + R * lane + r] = C[r];
          rec[rec_L(D) + R * lane + r] = L[r];
          rec[rec_mu(D) + R * lane + r] = mu[r];
        }
        if (lane == 0) {
          RecordHead* hd = reinterpret_cast<RecordHead*>(rec);
          hd->t = N;
          hd->mC = sc.mC;
          hd->EC = sc.EC;
          hd->CP = sc.CP;
          hd->etau = etau;
          hd->ml = sc.ml;
          hd->El = sc.El;
          hd->LP = sc.LP;
        }
      }
    }
    // no CTA of a LayerNorm cluster exits while another may still write its statistics
    if (clustered) cluster_sync_all();
    return;
  }

  // ---- encoder readout: every token against the full-sequence state ----
  __shared__ float fullsc[3];  // Et_N, P_N, m_N
  if (warp == 0 && lane == 0) {
    fullsc[0] = Et_run;
    fullsc[1] = P_run;
    fullsc[2] = m_run;
  }
  const float rN = __fdiv_rn(1.0f, (float)N);
  for (int t = 0; t < N; ++t) {
    __syncthreads();  // previous readout finished with qs / tc
    if (warp == 1) load_unit_row(q, t, qs);
    if (warp == 0 && lane == 0) {
      const float sig1 = sigmoid(g1[t]), sigh = sigmoid(gh[t]);
      tc.alpha = __fdiv_rn(sigh, fullsc[0]);
      tc.beta = __fmul_rn(__fsub_rn(sig1, sigh), rN);
      // the centred sums carry the -beta P / N and -sigh / N parts of gamma
      tc.gamma = a.g0 ? __fmul_rn(sigmoid(a.g0[row0 + t]), rN) : 0.0f;
      if (blockIdx.y == 0) {
        if (a.dbg_E) a.dbg_E[row0 + t] = fullsc[0];
        if (a.dbg_P) a.dbg_P[row0 + t] = fullsc[1];
        if (a.dbg_m) a.dbg_m[row0 + t] = fullsc[2];
      }
    }
    __syncthreads();
    float acc = 0.0f;
#pragma unroll
    for (int r = 0; r < RA; ++r) {
      const int ai = warp + 8 * r;
      const float comb = __fmaf_rn(tc.alpha, F[r], __fmaf_rn(tc.beta, G[r], __fmul_rn(tc.gamma, Hs[r])));
      acc = __fmaf_rn(qs[ai], comb, acc);
    }
    red[warp][lane] = acc;
    __syncthreads();
    if (warp == 7) {
      float o = red[0][lane];
#pragma unroll
      for (int w = 1; w < 8; ++w) o = __fadd_rn(o, red[w][lane]);
      emit(t, o);
    }
  }
  if (a.ln && warp == 7 && N > 0) ln_finish(N - 1);
  if (clustered) cluster_sync_all();
}

template <typename T>
cudaError_t launch_simt_typed(const FwdArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * a.H, a.d / 32, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = stream;
  // with the output LayerNorm the value slices of a head form one cluster
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = a.d / 32;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (a.ln && a.d > 32) ? 1 : 0;
  cudaError_t e;
  switch (a.d) {
    case 32: e = cudaLaunchKernelEx(&cfg, fwd_simt_kernel<T, 32>, a); break;
    case 64: e = cudaLaunchKernelEx(&cfg, fwd_simt_kernel<T, 64>, a); break;
    case 128: e = cudaLaunchKernelEx(&cfg, fwd_simt_kernel<T, 128>, a); break;
    default: return cudaErrorInvalidValue;
  }
  count_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
__global__ void state_init_kernel(void* state, const float* __restrict__ mu,
                                  const float* __restrict__ tau, int B, int H, int d) {
  const int bh = blockIdx.x;
  const int h = bh % H;
  float* rec = record_ptr(state, bh, d);
  const size_t nfl = record_bytes(d) / 4;
  for (size_t i = 8 + threadIdx.x; i < nfl; i += blockDim.x) rec[i] = 0.0f;
  __syncthreads();
  for (int i = threadIdx.x; i < d; i += blockDim.x) rec[rec_mu(d) + i] = mu[(size_t)h * d + i];
  if (threadIdx.x == 0) {
    RecordHead* hd = reinterpret_cast<RecordHead*>(rec);
    hd->t = 0;
    hd->mC = -INFINITY;
    hd->EC = 0.0f;
    hd->CP = 0.0f;
    hd->etau = expf(tau[h]);
    hd->ml = -INFINITY;
    hd->El = 0.0f;
    hd->LP = 0.0f;
  }
}

__global__ void state_header_kernel(void* state, int B, int H, int d, int dtype, int rope,
                                    float rope_base) {
  StateHeader* hdr = static_cast<StateHeader*>(state);
  int* w = reinterpret_cast<int*>(hdr);
  for (int i = threadIdx.x; i < 64; i += blockDim.x) w[i] = 0;
  __syncthreads();
  if (threadIdx.x == 0) {
    hdr->magic[0] = 'Z';
    hdr->magic[1] = 'S';
    hdr->magic[2] = 'P';
    hdr->magic[3] = '1';
    hdr->version = 1;
    hdr->B = B;
    hdr->H = H;
    hdr->d = d;
    hdr->dtype = dtype;
    hdr->rope = rope;
    hdr->rope_base = rope_base;
  }
}

// Rotary table [N][d/2] of (cos, sin) of pos * base^(-2a/d), computed in fp64.
__global__ void rope_table_kernel(float2* table, int N, int d, double base) {
  const int half = d / 2;
  const size_t total = (size_t)N * half;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int pos = (int)(i / half), pa = (int)(i % half);
    const double ang = (double)pos * pow(base, -2.0 * (double)pa / (double)d);
    double s, c;
    sincos(ang, &s, &c);
    table[i] = make_float2((float)c, (float)s);
  }
}

}  // namespace

// ------------------------------------------------------------------------------------------
// Scratch of the allocation-free forward (zeros_fwd_noalloc): the rotary table lives in this
// fixed device array instead of the library workspace.  Every device that loads the library
// holds it (1 MiB) until the process exits.
static __device__ __align__(256) float2 g_noalloc_rope[kNoAllocRopeEntries];

cudaError_t noalloc_rope_table(float2** table) {
  // Host code cannot use the array's name as a device address: ask the runtime for it, with the
  // calling device current.  The lookup is repeated on every call (it is a host-side query, not
  // stream work), so a context that was torn down and created again (cudaDeviceReset), which
  // may place the array elsewhere, is never served a stale address.
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_rope);
  if (e != cudaSuccess) return e;
  *table = static_cast<float2*>(p);
  return cudaSuccess;
}

cudaError_t launch_fwd_simt(const FwdArgs& a, cudaStream_t stream) {
  return a.dtype == 1 ? launch_simt_typed<float>(a, stream)
                      : launch_simt_typed<__nv_bfloat16>(a, stream);
}

cudaError_t launch_state_init(void* state, const float* mu, const float* tau, int B, int H, int d,
                              int dtype, int rope, float rope_base, cudaStream_t stream) {
  cudaError_t e = launch_state_header(state, B, H, d, dtype, rope, rope_base, stream);
  if (e != cudaSuccess) return e;
  if (B * H == 0) return cudaSuccess;
  state_init_kernel<<<B * H, 256, 0, stream>>>(state, mu, tau, B, H, d);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_state_header(void* state, int B, int H, int d, int dtype, int rope,
                                float rope_base, cudaStream_t stream) {
  state_header_kernel<<<1, 64, 0, stream>>>(state, B, H, d, dtype, rope, rope_base);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(float2* table, int N, int d, double base, cudaStream_t stream) {
  const size_t total = (size_t)N * (d / 2);
  const int blocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
  rope_table_kernel<<<blocks > 0 ? blocks : 1, 256, 0, stream>>>(table, N, d, base);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace zs
