/*
 * zeros.h - C ABI of the GB300 (sm_103a) hot path of ZeroS, zero-sum linear attention.
 *
 * What is computed (Paper-Notes "ZeroS: Zero-Sum Linear Attention for Efficient Transformers",
 * method details):
 *   deviation logits   s_i = -(1/sqrt d) u_i . ubar_i,
 *                      ubar_i = (e^tau mu + sum_{j<=i} u_j) / (e^tau + i)   ("deviation logits")
 *   zero-sum weights   w_{t,i} = sig1_t delta_{t,i}/t + sigh_t eps_{t,i}, sig = sigmoid(gate logit)
 *                      ("zero-order removal and zero-sum weights")
 *   angular factor     cos theta_{t,i} = q_hat_t R_{t-i} k_hat_i^T         ("radial-angular
 *                      decoupling", with RoPE)
 *   output             o_t = sum_i w_{t,i} cos theta_{t,i} v_i
 *                          = q_hat_t (alpha_t F_t + beta_t G_t + gamma_t H_t)  ("linear-time
 *                      prefix scan": E = sum e^s, P = sum s, F = sum e^s k_hat^T v,
 *                      G = sum s k_hat^T v, H = sum k_hat^T v)
 * with delta_{t,i} = s_i - P_t/t, eps_{t,i} = e^{s_i}/E_t - 1/t - delta_{t,i}/t, hence
 * alpha_t = sigh_t/E_t, beta_t = (sig1_t - sigh_t)/t, gamma_t = -(sig1_t - sigh_t) P_t/t^2 - sigh_t/t.
 * Causal (decoder) mode sums over i <= t; encoder mode sums over every token with t := N and
 * the full-sequence prior mean (page section "training strategy": both modes exist).
 * RoPE: half-split pairs (a, a + d/2), theta_a = base^(-2a/d), token t at position t - 1.
 *
 * Layouts (row-major, contiguous, all pointers are DEVICE pointers owned by the caller):
 *   q, k, v, u, out : [B, H, N, d]  bf16 (zeros_fwd) or the dtype given to zeros_fwd_ex
 *   g1, gh          : [B, H, N]     fp32 gate logits (sig1 = sigmoid(g1), sigh = sigmoid(gh))
 *   mu              : [H, d]        fp32 per-head prior mean
 *   tau             : [H]           fp32 per-head prior log-weight
 * Supported head dimensions: d in {32, 64, 128}.  Every pointer must be 16-byte aligned.
 *
 * Errors.  Argument checks run on the host before anything is launched and return a nonzero
 * zeros_status without touching the GPU.  Conditions found on the device (a non-finite logit,
 * an exponent out of fp32 range, a bounded wait that gave up) are recorded in a per-device
 * status word; zeros_get_status() synchronises the stream and returns and clears it.  Outputs
 * are unspecified when a call or the status word reports an error.  All launches are
 * asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *
 * Memory.  The library allocates nothing per call once warm: it keeps one lazily created,
 * per-device workspace that only grows (growing it waits for the device) and is released at
 * process exit: rotary tables; for the chunked causal path 16*B*H*N bytes of per-token
 * scalars; the backward and ZeroS-SM scratches described at those calls.  Code that captures
 * calls into a CUDA graph makes one call of the same or larger size before the capture.  The
 * workspace is shared by every stream of the device: calls on different streams must not
 * overlap on the GPU (order them with events), or they overwrite each other's scratch.
 */
#ifndef ZEROS_H
#define ZEROS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ZEROS_OK = 0,
  ZEROS_ERR_INVALID = 1,     /* bad argument: null pointer, negative size, misalignment     */
  ZEROS_ERR_UNSUPPORTED = 2, /* well-formed but not supported (d not in {32,64,128}, ...)   */
  ZEROS_ERR_RANGE = 3,       /* device: non-finite logit or exponent outside fp32 range     */
  ZEROS_ERR_TIMEOUT = 4,     /* device: a bounded wait gave up                              */
  ZEROS_ERR_CUDA = 5         /* a CUDA runtime call failed (see zeros_last_error_message)   */
} zeros_status;

typedef enum { ZEROS_BF16 = 0, ZEROS_F32 = 1 } zeros_dtype;

/* Implementation selector for zeros_fwd_ex (all produce the same result up to rounding). */
typedef enum {
  ZEROS_PATH_AUTO = 0,  /* chunked tensor-core scan where available, else the SIMT scan      */
  ZEROS_PATH_SIMT = 1,  /* token-sequential CUDA-core scan (fp32 and bf16 inputs)            */
  ZEROS_PATH_CHUNK = 2  /* chunked tcgen05/TMEM scan (bf16 inputs, causal): a scalar pass
                           (per-token logits and prefix scalars), then the chunk kernel         */
} zeros_path;

/*
 * Forward pass over [B, H, N, d] bf16 inputs, bf16 output, rotary base 10000.
 * causal = 1: decoder mode (prefix sums); causal = 0: encoder mode (full-sequence sums).
 * rope   = 1: rotary positions in the angular factor.
 * B, H or N equal to 0 is a valid empty call (returns ZEROS_OK, launches nothing).
 */
int zeros_fwd(const void* q, const void* k, const void* v, const void* u, const float* g1,
              const float* gh, const float* mu, const float* tau, void* out, int B, int H, int N,
              int d, int causal, int rope, void* stream);

/*
 * zeros_fwd with every option.
 *   g0          : nullable fp32 [B, H, N]: zero-order gate logits of a first layer (Paper-Notes
 *                 "ZeroS", zero-order removal: the first layer may keep the zero-order term).
 *                 Every weight gains sigmoid(g0_t) / t (encoder: / N), so the weights of
 *                 query t sum to sigmoid(g0_t) instead of 0.  NULL: no zero-order term (the
 *                 pages' default).
 *   dtype       : ZEROS_BF16 or ZEROS_F32 for q, k, v, u and out.
 *   rope_base   : rotary base (> 0) when rope = 1.
 *   path        : a zeros_path value.
 *   final_state : nullable; causal only.  A state blob of zeros_state_bytes(B, H, d) bytes that
 *                 receives the recurrent state after the N tokens (prefill for
 *                 zeros_decode_step).  It records dtype, rope and rope_base.
 *   dbg_s, dbg_E, dbg_P, dbg_m : nullable fp32 [B, H, N].  Per token: the logit s_t, the
 *                 scaled prefix sum E_t e^{-m_t}, the prefix sum P_t and the running maximum
 *                 m_t = max_{i<=t} s_i (encoder: the full-sequence values).  These four are
 *                 bit-identical to those zeros_decode_step_ex reports for the same tokens.
 */
int zeros_fwd_ex(const void* q, const void* k, const void* v, const void* u, const float* g1,
                 const float* gh, const float* g0, const float* mu, const float* tau, void* out,
                 int B, int H,
                 int N, int d, int causal, int rope, int dtype, float rope_base, int path,
                 void* final_state, float* dbg_s, float* dbg_E, float* dbg_P, float* dbg_m,
                 void* stream);

/*
 * Forward with a fused output LayerNorm (Paper-Notes "ZeroS", ablation table: removing the
 * LayerNorm costs accuracy; highlights: LayerNorm supersedes the 1/sqrt(t) Lipschitz decay.
 * The pages do not place it; read here as the normalisation of each head's output row):
 *   y_t = (o_t - mean(o_t)) / sqrt(var(o_t) + ln_eps) * ln_w[h] + ln_b[h]
 * over the d columns of o_t, var the population variance, before the output is rounded to
 * its dtype.  Same computation, layouts and other arguments as zeros_fwd_ex (without debug
 * outputs); final_state (prefill) holds the un-normalised scan state as there.
 *   ln_w, ln_b : nullable fp32 [H, d] gain and bias (NULL: 1 and 0), 16-byte aligned
 *   ln_eps     : finite, >= 0
 * On the GPU the d / 32 value slices of a head run as one thread-block cluster and exchange
 * their rows' statistics through distributed shared memory.
 */
int zeros_fwd_ln(const void* q, const void* k, const void* v, const void* u, const float* g1,
                 const float* gh, const float* g0, const float* mu, const float* tau,
                 const float* ln_w, const float* ln_b, float ln_eps, void* out, int B, int H,
                 int N, int d, int causal, int rope, int dtype, float rope_base, int path,
                 void* final_state, void* stream);

/*
 * ZeroS-SM, the quadratic variant (Paper-Notes "ZeroS", linear-time prefix scan: the same
 * zero-sum reweighting applied to standard softmax attention; its formula sits in an appendix
 * the pages do not include).  Reading: logits s_{t,i} = q_t k_i^T / sqrt(d) with raw q, k
 * (rotated to their positions when rope = 1), and per query t over its keys i (i <= t when
 * causal = 1, every key with t := N when causal = 0)
 *   w_{t,i} = sig1_t delta_{t,i}/t + sigh_t eps_{t,i} (+ sig0_t/t),  o_t = sum_i w_{t,i} v_i,
 *   delta_{t,i} = s_{t,i} - (1/t) sum_j s_{t,j},  eps_{t,i} = softmax_{t,i} - 1/t - delta_{t,i}/t.
 *   q, k, v, out : [B, H, N, d] bf16 (dtype must be ZEROS_BF16), d in {64, 128}
 *   g1, gh, g0   : fp32 [B, H, N] gate logits (g0 nullable: the zero-order gate)
 *   N <= 8388480.  O(N^2 d) work on the tensor cores; with rope = 1 the library rotates q and k
 *   into a per-device scratch of 4*B*H*N*d bytes (grown on demand; growing it waits for the
 *   device) and keeps a rotary table as zeros_fwd_ex does.
 */
int zeros_sm_fwd(const void* q, const void* k, const void* v, const float* g1, const float* gh,
                 const float* g0, void* out, int B, int H, int N, int d, int causal, int rope,
                 int dtype, float rope_base, void* stream);

/*
 * Allocation-free forward (the pages have no counterpart: this entry point exists for callers
 * that must not allocate device memory themselves or through this library, for example code
 * whose device memory is all handed out up front by its own allocator, or a runtime that forbids
 * cudaMalloc once it is serving).  Same computation and layouts as zeros_fwd_ex on the
 * token-sequential path (ZEROS_PATH_SIMT), without final state or debug outputs.
 *   - It calls no cudaMalloc / cudaFree and no allocating routine.  Its only scratch, the rotary
 *     (cos, sin) table, lives in a fixed 1 MiB device array compiled into the library, which every
 *     device that loads the library holds until the process exits; with rope = 1 it needs
 *     N * d / 2 <= 131072 and returns ZEROS_ERR_UNSUPPORTED beyond that.
 *   - Every call looks up the array's device address on the current device
 *     (cudaGetSymbolAddress), so a context that was reset and created again is served its new
 *     address.  The first call on a device may load the library's device code for that
 *     device: make that first call before any stream capture.
 *   - Every call rewrites the shared table, so calls that overlap on the GPU (different streams
 *     at the same time) race; serialise them.
 *   - status: nullable device int, caller-owned.  It is zeroed on `stream` at the start of the
 *     call and receives the first device-side error (ZEROS_ERR_RANGE ...); read it after the
 *     stream has finished.  The library's own status word (zeros_get_status) is not used.
 */
int zeros_fwd_noalloc(const void* q, const void* k, const void* v, const void* u,
                      const float* g1, const float* gh, const float* mu, const float* tau,
                      void* out, int B, int H, int N, int d, int causal, int rope, int dtype,
                      float rope_base, int* status, void* stream);

/*
 * Backward pass of the causal forward (training): gradients of L = sum(out * dout) with respect
 * to every input.  Differentiates the pages' five-state scan (Paper-Notes "ZeroS", method
 * details: deviation logits, zero-sum weights, radial-angular decoupling, linear-time prefix
 * scan); the pages give no backward, this is the derivative of that definition.
 *   q, k, v, u, dout          : [B, H, N, d] in `dtype` (ZEROS_BF16 or ZEROS_F32)
 *   g1, gh, mu, tau, g0       : as in zeros_fwd_ex (g0 nullable)
 *   dq, dk, dv, du            : [B, H, N, d] fp32, written
 *   dg1, dgh                  : [B, H, N] fp32, written;  dg0: nullable, needs g0
 *   dmu [H, d], dtau [H]      : fp32, overwritten with the sums over the batch
 * Causal mode only.  The library keeps a per-device scratch of B*H*N*(8+d)*4 bytes for the
 * pass (grown on demand; growing it waits for the device).  Gradients are reduced in fp32;
 * dmu and dtau are summed over the batch with atomic adds (order not fixed).
 */
int zeros_bwd(const void* q, const void* k, const void* v, const void* u, const float* g1,
              const float* gh, const float* g0, const float* mu, const float* tau,
              const void* dout, float* dq, float* dk, float* dv, float* du, float* dg1,
              float* dgh, float* dg0, float* dmu, float* dtau, int B, int H, int N, int d,
              int rope, int dtype, float rope_base, void* stream);

/* zeros_bwd with an implementation path (a zeros_path value): ZEROS_PATH_SIMT = the
 * token-sequential kernel (any d); ZEROS_PATH_CHUNK = the chunk-parallel kernels (d = 64 only,
 * else ZEROS_ERR_UNSUPPORTED): a forward launch supplies the per-token scalars, then per chunk
 * of 64 tokens the intra-chunk products and the inter-chunk terms from stored chunk-start and
 * suffix states (scratch of about B*H*N*(6 d + 8)*4 + 24 B*H*ceil(N/64)*d*d bytes);
 * ZEROS_PATH_AUTO = the chunked kernels where supported.  Both reduce in fp32. */
int zeros_bwd_ex(const void* q, const void* k, const void* v, const void* u, const float* g1,
                 const float* gh, const float* g0, const float* mu, const float* tau,
                 const void* dout, float* dq, float* dk, float* dv, float* du, float* dg1,
                 float* dgh, float* dg0, float* dmu, float* dtau, int B, int H, int N, int d,
                 int rope, int dtype, float rope_base, int path, void* stream);

/*
 * Recurrent state ("the state is the checkpoint").  Size in bytes of the blob for B x H
 * sequences of head dimension d (0 for unsupported d).  Layout: a 256-byte header
 * {magic "ZSP1", version, B, H, d, dtype, rope, rope_base} followed by B*H records of
 * zeros_state_record_bytes(d) bytes; record (b, h) at index b*H + h holds
 *   int32 t (tokens seen), then the running scalars in the library's blocked order (tokens in
 *   blocks of 32: a carry at the end of the last completed block plus a local value for the
 *   current block): fp32 mC, EC, CP (carries of the running max m, of E e^{-m} and of P),
 *   fp32 e^tau, fp32 ml, El, LP (block-local running max, scaled exp-sum and logit sum),
 *   fp32 C[d] (carry of the running sum of u), fp32 L[d] (block-local sum of u), fp32 mu[d],
 *   fp32 F~[d][d] (= F e^{-m}), fp32 G[d][d], fp32 H[d][d]   (row a = key dim, col j = value dim)
 * padded to a multiple of 256 bytes.  The blob may be copied, saved and restored byte-wise.
 */
size_t zeros_state_bytes(int B, int H, int d);
size_t zeros_state_record_bytes(int d);

/* Empty state (t = 0) for B x H sequences with prior mu [H, d] and tau [H] (device fp32). */
int zeros_state_init(void* state, const float* mu, const float* tau, int B, int H, int d,
                     int dtype, int rope, float rope_base, void* stream);

/*
 * One recurrent-inference step (the linear-time prefix scan applied to one new token) for
 * every sequence in the state: q, k, v, u [B, H, d] and out [B, H, d] in the state's dtype,
 * g1, gh [B, H] fp32.  Advances t by one; the token's rotary position is the old t.
 * The state must come from zeros_state_init or zeros_fwd_ex(final_state) in this process;
 * otherwise its 256-byte header is read once from the device (a synchronous copy).
 */
int zeros_decode_step(void* state, const void* q, const void* k, const void* v, const void* u,
                      const float* g1, const float* gh, void* out, void* stream);

/* As zeros_decode_step with explicit dimensions (no header lookup), the zero-order gate g0
 * (nullable fp32 [B, H], as in zeros_fwd_ex) and per-token debug outputs dbg_s, dbg_E, dbg_P,
 * dbg_m (nullable fp32 [B, H]) as in zeros_fwd_ex. */
int zeros_decode_step_ex(void* state, int B, int H, int d, const void* q, const void* k,
                         const void* v, const void* u, const float* g1, const float* gh,
                         const float* g0,
                         void* out, float* dbg_s, float* dbg_E, float* dbg_P, float* dbg_m,
                         void* stream);

/* zeros_decode_step_ex with the fused output LayerNorm of zeros_fwd_ln (ln_w, ln_b nullable
 * fp32 [H, d]; ln_eps finite, >= 0) and no debug outputs.  The state is not affected by it. */
int zeros_decode_step_ln(void* state, int B, int H, int d, const void* q, const void* k,
                         const void* v, const void* u, const float* g1, const float* gh,
                         const float* g0, const float* ln_w, const float* ln_b, float ln_eps,
                         void* out, void* stream);

/* Synchronises `stream`, then returns and clears the current device's status word. */
int zeros_get_status(void* stream);

/* Static description of a status code. */
const char* zeros_status_string(int status);

/* Detail of the last host-side error on this thread ("" if none). */
const char* zeros_last_error_message(void);

/* ABI version of this library (major * 100 + minor). */
int zeros_version(void);

/* Number of CUDA kernels this process has launched through the library so far (all devices,
 * all entry points).  Used by benchmarks to count device work; never reset. */
unsigned long long zeros_kernel_launches(void);

/* Testing hook for the failure path of the d = 64 tensor-core forward (the bf16 causal
 * forward at d = 64 on the chunked path).  Every wait of that kernel on another warp's
 * progress is bounded; when one gives up the kernel records ZEROS_ERR_TIMEOUT, its other warps
 * leave their loops, it waits for its own copies and tensor-core work still in flight, frees
 * its tensor memory and returns, so that the context stays usable.
 *   wait_limit_cycles  > 0: bound of each such wait in SM clock cycles for later launches;
 *                      0: the default (2^32 cycles, about two seconds).
 *   skip_one_arrive    nonzero: in later launches one warp of every CTA withholds its arrival
 *                      on the barrier that releases the first S V product, so that the wait
 *                      for it runs out (and everything after it is abandoned).
 * Both are process-wide settings, off by default; set them only while no forward runs on any
 * thread.  Returns ZEROS_OK, or ZEROS_ERR_INVALID for a negative limit. */
int zeros_debug_walk(long long wait_limit_cycles, int skip_one_arrive);

#ifdef __cplusplus
}
#endif

#endif /* ZEROS_H */
