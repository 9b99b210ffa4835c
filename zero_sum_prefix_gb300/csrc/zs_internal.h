// Host-side declarations shared by the translation units of the ZeroS library.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace zs {

// Everything a forward launch needs; pointers are device pointers.
struct FwdArgs {
  const void *q, *k, *v, *u;
  const float *g1, *gh, *mu, *tau;
  const float* g0;  // nullable: zero-order gate logits [B,H,N]
  void* out;
  int B, H, N, d;
  int causal, rope, dtype;
  float rope_base;
  const float2* rope_table;  // [N][d/2] (cos, sin) when rope, else null
  void* final_state;         // nullable (causal only)
  float *dbg_s, *dbg_E, *dbg_P, *dbg_m;
  int* status;               // device status word
  int ln;                    // output LayerNorm over each head's d columns
  const float *ln_w, *ln_b;  // nullable [H,d] gain and bias
  float ln_eps;
  // chunked path: per-token (s, m, Et, P) of the blocked contract, [B*H, N], written by
  // launch_fwd_scalars before the chunk kernel reads it
  float4* scal;
  // nullable: per sequence and scalar-pass CTA, the largest |s| of its tokens, [B*H, 8]
  float* smax;
};

struct DecodeArgs {
  void* state;
  const void *q, *k, *v, *u;
  const float *g1, *gh;
  const float* g0;  // nullable: zero-order gate logits [B,H]
  void* out;
  int B, H, d, dtype, rope;
  float rope_base;
  float *dbg_s, *dbg_E, *dbg_P, *dbg_m;
  int* status;
  int ln;                    // output LayerNorm as in FwdArgs
  const float *ln_w, *ln_b;
  float ln_eps;
};

struct BwdArgs {
  const void *q, *k, *v, *u, *dout;  // [B,H,N,d] input dtype
  const float *g1, *gh, *g0;         // [B,H,N] (g0 nullable)
  const float *mu, *tau;             // [H,d], [H]
  float *dq, *dk, *dv, *du;          // [B,H,N,d] fp32
  float *dg1, *dgh, *dg0;            // [B,H,N] fp32 (dg0 nullable)
  float *dmu, *dtau;                 // [H,d], [H] fp32, accumulated (zeroed by the host)
  float* scratch;                    // bwd_scratch_bytes
  const float2* rope_table;          // [N][d/2] when rope
  int B, H, N, d, rope, dtype;
  int* status;
};

// ZeroS-SM (quadratic variant): bf16 q, k (already rotated when rotary positions are used),
// v [B,H,N,d]; fp32 gates [B,H,N]; bf16 out.
struct SmArgs {
  const void *q, *k, *v;
  const float *g1, *gh, *g0;  // g0 nullable
  void* out;
  int B, H, N, d, causal;
  int* status;
  // d = 64: per 128-token tile, [B*H][tiles][kSmStat] fp32: the column sums of k as the kernel
  // reads it (0..63), the largest row norm of k (64), the column sums of v (68..131), the norm
  // of each row of q as the kernel reads it (132..259); written by launch_sm_prep
  const float* kstat;
};
constexpr int kSmStat = 260;

// Counts every kernel launch the library issues (zs_api.cu).
void count_launches(unsigned n);

// zs_simt.cu
cudaError_t launch_fwd_simt(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_state_init(void* state, const float* mu, const float* tau, int B, int H, int d,
                              int dtype, int rope, float rope_base, cudaStream_t stream);
cudaError_t launch_state_header(void* state, int B, int H, int d, int dtype, int rope,
                                float rope_base, cudaStream_t stream);
cudaError_t launch_rope_table(float2* table, int N, int d, double base, cudaStream_t stream);

// Fixed scratch of the allocation-free forward: (cos, sin) entries for N * d/2 <= this bound.
constexpr size_t kNoAllocRopeEntries = size_t(1) << 17;
// Device address of that scratch on the current device (looked up on every call).
cudaError_t noalloc_rope_table(float2** table);

// zs_chunk.cu: the chunked forward (bf16, causal; d = 128, and d = 64 with the fused output
// LayerNorm).  a.scal must hold the per-token scalars (launch_fwd_scalars on the same stream
// first).  chunk_supported tells whether the chunked path (this kernel or zs_walk.cu) exists.
bool chunk_supported(int d, int dtype, int causal);
cudaError_t launch_fwd_chunk(const FwdArgs& a, cudaStream_t stream);

// zs_walk.cu: the causal forward for d = 64 (bf16): one CTA per (sequence, segment), all 64
// value columns of a head in one CTA.  a.scal must hold the per-token scalars; with rope, `ang`
// holds walk_angle_floats(N) floats written by launch_walk_angles.  nseg_max bounds the number
// of segments per sequence.
bool walk_supported(int d, int dtype, int causal);
size_t walk_angle_floats(int N);
cudaError_t launch_walk_angles(float* tab, int N, double base, cudaStream_t stream);
cudaError_t launch_fwd_walk(const FwdArgs& a, const float* ang, int nseg_max,
                            cudaStream_t stream);
// Testing hook of zeros_debug_walk: the wait bound of later walk launches (0 = default) and
// whether one warp per CTA withholds its first arrival on the S-tile barrier.
void set_walk_debug(long long wait_limit_cycles, int skip_one_arrive);

// zs_scalars.cu: per-token (s, m, Et, P) of every sequence into scal ([B*H, N] float4), the
// largest |s| per sequence and CTA into a.smax when given ([B*H, kScalarCtas]), the debug
// scalars and the scalar part of the final state when asked for (d in {64, 128}).
constexpr int kScalarCtas = 8;
cudaError_t launch_fwd_scalars(const FwdArgs& a, float4* scal, cudaStream_t stream);

// zs_backward.cu
size_t bwd_scratch_bytes(int B, int H, int N, int d);
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream);

// zs_decode.cu
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

// zs_backward_chunk.cu: chunk-parallel backward (d = 64).  The scratch starts with the forward
// scalars s, E e^{-m}, P, m ([B*H*N] each), which the caller fills by a forward launch with
// those debug outputs.
bool bwd_chunk_supported(int d);
size_t bwd_chunk_scratch_bytes(int B, int H, int N, int d);
cudaError_t launch_bwd_chunk(const BwdArgs& a, float* scratch, cudaStream_t stream);

// zs_encoder.cu: encoder-mode forward in 64-token tiles (d = 64; no debug outputs)
bool enc_supported(int d);
cudaError_t launch_fwd_encoder(const FwdArgs& a, cudaStream_t stream);

// zs_sm.cu
bool sm_supported(int d, int dtype);
cudaError_t launch_sm(const SmArgs& a, cudaStream_t stream);
cudaError_t launch_sm_rotate(const void* q, const void* k, void* yq, void* yk,
                             const float2* table, int BH, int N, int d, cudaStream_t stream);
// d = 64: the key-tile statistics of SmArgs::kstat, and with a rotary table also the rotated q
// and k (into yq, yk; as launch_sm_rotate writes them), in one pass; a wait that gives up is
// reported in *status.
cudaError_t launch_sm_prep(const void* q, const void* k, const void* v, void* yq, void* yk,
                           const float2* table, float* kstat, int* status, int BH, int N,
                           cudaStream_t stream);

}  // namespace zs
