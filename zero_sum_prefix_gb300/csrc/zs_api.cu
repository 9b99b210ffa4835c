// Host side of the ZeroS C ABI (include/zeros.h): argument validation, the per-device
// workspace (status word, rotary tables), the state registry and the stream-ordered launches.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>

#include "zeros.h"
#include "zs_common.cuh"
#include "zs_internal.h"

namespace zs {
namespace {

thread_local std::string g_last_error;
std::atomic<unsigned long long> g_launches{0};

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(ZEROS_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

struct DeviceWorkspace {
  int* status = nullptr;
  float* bwd = nullptr;  // backward scratch (per-token scalars and prior means)
  size_t bwd_bytes = 0;
  void* sm = nullptr;     // ZeroS-SM scratch (rotated q and k)
  size_t sm_bytes = 0;
  void* fwd = nullptr;    // chunked forward scratch (per-token scalars)
  size_t fwd_bytes = 0;
  float* wang = nullptr;  // rotary angles of the d = 64 walk (frequencies, chunk base angles)
  size_t wang_floats = 0;
  int wang_N = 0;
  float wang_base = 0.0f;
  float2* rope = nullptr;
  size_t rope_entries = 0;  // capacity in float2
  int rope_N = 0, rope_d = 0;
  float rope_base = 0.0f;
};

std::mutex g_mutex;
std::unordered_map<int, DeviceWorkspace> g_ws;

struct StateInfo {
  int B, H, d, dtype, rope;
  float rope_base;
};
std::unordered_map<const void*, StateInfo> g_states;

int current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  return ZEROS_OK;
}

// Per-device workspace with the status word (allocated once, zeroed).
int workspace(DeviceWorkspace** out) {
  int dev;
  if (int rc = current_device(&dev)) return rc;
  std::lock_guard<std::mutex> lk(g_mutex);
  DeviceWorkspace& ws = g_ws[dev];
  if (!ws.status) {
    cudaError_t e = cudaMalloc(&ws.status, 256);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(status)");
    e = cudaMemset(ws.status, 0, 256);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(status)");
  }
  *out = &ws;
  return ZEROS_OK;
}

// Rotary (cos, sin) table for positions [0, N) and head dimension d, built on `stream`.
int rope_table(DeviceWorkspace* ws, int N, int d, float base, cudaStream_t stream,
               const float2** table) {
  std::lock_guard<std::mutex> lk(g_mutex);
  if (ws->rope && ws->rope_d == d && ws->rope_base == base && ws->rope_N >= N) {
    *table = ws->rope;
    return ZEROS_OK;
  }
  const int n_new = N > 0 ? N : 1;
  const size_t need = (size_t)n_new * (size_t)(d / 2);
  if (ws->rope) {
    // Work already queued (on any stream) may still read the current table.
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  }
  if (need > ws->rope_entries) {
    if (ws->rope) cudaFree(ws->rope);
    ws->rope = nullptr;
    ws->rope_entries = 0;
    cudaError_t e = cudaMalloc(&ws->rope, need * sizeof(float2));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(rope table)");
    ws->rope_entries = need;
  }
  cudaError_t e = launch_rope_table(ws->rope, n_new, d, (double)base, stream);
  if (e != cudaSuccess) return cuda_fail(e, "rope table launch");
  ws->rope_N = n_new;
  ws->rope_d = d;
  ws->rope_base = base;
  *table = ws->rope;
  return ZEROS_OK;
}

// Rotary angle table of the d = 64 walk for N tokens and the given base, built on `stream`.
int walk_angles(DeviceWorkspace* ws, int N, float base, cudaStream_t stream, const float** tab) {
  std::lock_guard<std::mutex> lk(g_mutex);
  if (ws->wang && ws->wang_base == base && ws->wang_N >= N) {
    *tab = ws->wang;
    return ZEROS_OK;
  }
  const size_t need = walk_angle_floats(N);
  if (ws->wang) {
    // Work already queued (on any stream) may still read the current table.
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  }
  if (need > ws->wang_floats) {
    if (ws->wang) cudaFree(ws->wang);
    ws->wang = nullptr;
    ws->wang_floats = 0;
    cudaError_t e = cudaMalloc(&ws->wang, need * sizeof(float));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(walk angle table)");
    ws->wang_floats = need;
  }
  cudaError_t e = launch_walk_angles(ws->wang, N, (double)base, stream);
  if (e != cudaSuccess) return cuda_fail(e, "walk angle table launch");
  ws->wang_N = N;
  ws->wang_base = base;
  *tab = ws->wang;
  return ZEROS_OK;
}

// Upper bound on the segments per sequence of the d = 64 walk: ZEROS_MAX_SEGMENTS (1 to 4)
// when set, else 4.
int walk_max_segments() {
  const char* env = getenv("ZEROS_MAX_SEGMENTS");
  if (!env) return 4;
  const int v = atoi(env);
  return v < 1 ? 1 : (v > 4 ? 4 : v);
}

// Backward scratch of at least `bytes`, grown on demand (after the device has drained: queued
// work may still use the old buffer).
int bwd_scratch(DeviceWorkspace* ws, size_t bytes, float** out) {
  std::lock_guard<std::mutex> lk(g_mutex);
  if (bytes > ws->bwd_bytes) {
    if (ws->bwd) {
      cudaError_t e = cudaDeviceSynchronize();
      if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
      cudaFree(ws->bwd);
    }
    ws->bwd = nullptr;
    ws->bwd_bytes = 0;
    cudaError_t e = cudaMalloc(&ws->bwd, bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(backward scratch)");
    ws->bwd_bytes = bytes;
  }
  *out = ws->bwd;
  return ZEROS_OK;
}

// ZeroS-SM scratch of at least `bytes` (grown like the backward scratch).
int sm_scratch(DeviceWorkspace* ws, size_t bytes, void** out) {
  std::lock_guard<std::mutex> lk(g_mutex);
  if (bytes > ws->sm_bytes) {
    if (ws->sm) {
      cudaError_t e = cudaDeviceSynchronize();
      if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
      cudaFree(ws->sm);
    }
    ws->sm = nullptr;
    ws->sm_bytes = 0;
    cudaError_t e = cudaMalloc(&ws->sm, bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(ZeroS-SM scratch)");
    ws->sm_bytes = bytes;
  }
  *out = ws->sm;
  return ZEROS_OK;
}

// Chunked forward scratch of at least `bytes` (grown like the backward scratch).
int fwd_scratch(DeviceWorkspace* ws, size_t bytes, void** out) {
  std::lock_guard<std::mutex> lk(g_mutex);
  if (bytes > ws->fwd_bytes) {
    if (ws->fwd) {
      cudaError_t e = cudaDeviceSynchronize();
      if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
      cudaFree(ws->fwd);
    }
    ws->fwd = nullptr;
    ws->fwd_bytes = 0;
    cudaError_t e = cudaMalloc(&ws->fwd, bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(forward scratch)");
    ws->fwd_bytes = bytes;
  }
  *out = ws->fwd;
  return ZEROS_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_ptr(const void* p, const char* name) {
  if (!p) return fail(ZEROS_ERR_INVALID, std::string(name) + " is null");
  if (!aligned16(p)) return fail(ZEROS_ERR_INVALID, std::string(name) + " is not 16-byte aligned");
  return ZEROS_OK;
}

int check_opt_ptr(const void* p, const char* name) {
  if (p && !aligned16(p))
    return fail(ZEROS_ERR_INVALID, std::string(name) + " is not 16-byte aligned");
  return ZEROS_OK;
}

int check_dims(int B, int H, int N, int d) {
  if (B < 0 || H < 0 || N < 0) return fail(ZEROS_ERR_INVALID, "negative B, H or N");
  if (d != 32 && d != 64 && d != 128)
    return fail(ZEROS_ERR_UNSUPPORTED, "head dimension d must be 32, 64 or 128");
  const unsigned long long bh = (unsigned long long)B * (unsigned long long)H;
  if (bh > 0x7fffffffull) return fail(ZEROS_ERR_INVALID, "B*H exceeds 2^31-1");
  if (bh * (unsigned long long)N * (unsigned long long)d > (1ull << 50))
    return fail(ZEROS_ERR_INVALID, "B*H*N*d exceeds 2^50 elements");
  if ((unsigned long long)N >= (1ull << 24))
    return fail(ZEROS_ERR_UNSUPPORTED, "N must be below 2^24 (token counts are exact in fp32)");
  return ZEROS_OK;
}

int check_dtype(int dtype) {
  if (dtype != ZEROS_BF16 && dtype != ZEROS_F32) return fail(ZEROS_ERR_INVALID, "unknown dtype");
  return ZEROS_OK;
}

}  // namespace

void count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

}  // namespace zs

using namespace zs;

extern "C" {

int zeros_version(void) { return 100; }

unsigned long long zeros_kernel_launches(void) { return g_launches.load(); }

int zeros_debug_walk(long long wait_limit_cycles, int skip_one_arrive) {
  if (wait_limit_cycles < 0) return fail(ZEROS_ERR_INVALID, "negative wait limit");
  set_walk_debug(wait_limit_cycles, skip_one_arrive);
  return ZEROS_OK;
}

const char* zeros_status_string(int status) {
  switch (status) {
    case ZEROS_OK: return "ok";
    case ZEROS_ERR_INVALID: return "invalid argument";
    case ZEROS_ERR_UNSUPPORTED: return "unsupported configuration";
    case ZEROS_ERR_RANGE: return "value out of range on the device";
    case ZEROS_ERR_TIMEOUT: return "a bounded device wait gave up";
    case ZEROS_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}

const char* zeros_last_error_message(void) { return g_last_error.c_str(); }

size_t zeros_state_record_bytes(int d) {
  if (d != 32 && d != 64 && d != 128) return 0;
  return record_bytes(d);
}

size_t zeros_state_bytes(int B, int H, int d) {
  if (B < 0 || H < 0 || (d != 32 && d != 64 && d != 128)) return 0;
  return state_bytes(B, H, d);
}

static int check_ln(int ln, const float* ln_w, const float* ln_b, float ln_eps) {
  if (!ln) return ZEROS_OK;
  if (!(ln_eps >= 0.0f && ln_eps <= 3.0e38f))
    return fail(ZEROS_ERR_INVALID, "ln_eps must be finite and >= 0");
  if (int rc = check_opt_ptr(ln_w, "ln_w")) return rc;
  return check_opt_ptr(ln_b, "ln_b");
}

static int fwd_impl(const void* q, const void* k, const void* v, const void* u, const float* g1,
                    const float* gh, const float* g0, const float* mu, const float* tau,
                    void* out, int B, int H, int N, int d, int causal, int rope, int dtype,
                    float rope_base, int path, void* final_state, float* dbg_s, float* dbg_E,
                    float* dbg_P, float* dbg_m, int ln, const float* ln_w, const float* ln_b,
                    float ln_eps, void* stream) {
  g_last_error.clear();
  if (int rc = check_dims(B, H, N, d)) return rc;
  if (int rc = check_ln(ln, ln_w, ln_b, ln_eps)) return rc;
  if (int rc = check_dtype(dtype)) return rc;
  if (causal != 0 && causal != 1) return fail(ZEROS_ERR_INVALID, "causal must be 0 or 1");
  if (rope != 0 && rope != 1) return fail(ZEROS_ERR_INVALID, "rope must be 0 or 1");
  if (rope && !(rope_base > 0.0f)) return fail(ZEROS_ERR_INVALID, "rope_base must be > 0");
  if (path != ZEROS_PATH_AUTO && path != ZEROS_PATH_SIMT && path != ZEROS_PATH_CHUNK)
    return fail(ZEROS_ERR_INVALID, "unknown path");
  if (final_state && !causal)
    return fail(ZEROS_ERR_INVALID, "final_state is only defined for the causal mode");
  const char* names[] = {"q", "k", "v", "u", "g1", "gh", "mu", "tau", "out"};
  const void* ptrs[] = {q, k, v, u, g1, gh, mu, tau, out};
  const bool empty = (long long)B * H * N == 0;
  if (!empty)
    for (int i = 0; i < 9; ++i)
      if (int rc = check_ptr(ptrs[i], names[i])) return rc;
  if (int rc = check_opt_ptr(final_state, "final_state")) return rc;
  if (int rc = check_opt_ptr(g0, "g0")) return rc;
  if (int rc = check_opt_ptr(dbg_s, "dbg_s")) return rc;
  if (int rc = check_opt_ptr(dbg_E, "dbg_E")) return rc;
  if (int rc = check_opt_ptr(dbg_P, "dbg_P")) return rc;
  if (int rc = check_opt_ptr(dbg_m, "dbg_m")) return rc;
  const bool chunk_ok = chunk_supported(d, dtype, causal);
  if (path == ZEROS_PATH_CHUNK && !chunk_ok)
    return fail(ZEROS_ERR_UNSUPPORTED,
                "the chunked tensor-core path needs bf16, causal mode and d in {64, 128}");
  const bool use_chunk = chunk_ok && path != ZEROS_PATH_SIMT;
  // encoder mode: the tiled kernel, unless the token-sequential path or its debug scalars are
  // asked for
  const bool use_enc = !causal && enc_supported(d) && path != ZEROS_PATH_SIMT && !dbg_s &&
                       !dbg_E && !dbg_P && !dbg_m;
  if (B == 0 || H == 0 || (N == 0 && !final_state)) return ZEROS_OK;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DeviceWorkspace* ws;
  if (int rc = workspace(&ws)) return rc;

  if (final_state) {
    if (!mu || !tau) return fail(ZEROS_ERR_INVALID, "mu/tau are null");
    cudaError_t e = launch_state_init(final_state, mu, tau, B, H, d, dtype, rope, rope_base, st);
    if (e != cudaSuccess) return cuda_fail(e, "state init launch");
    std::lock_guard<std::mutex> lk(g_mutex);
    g_states[final_state] = StateInfo{B, H, d, dtype, rope, rope_base};
  }
  if (N == 0) return ZEROS_OK;

  FwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.u = u;
  a.g1 = g1;
  a.gh = gh;
  a.g0 = g0;
  a.mu = mu;
  a.tau = tau;
  a.out = out;
  a.B = B;
  a.H = H;
  a.N = N;
  a.d = d;
  a.causal = causal;
  a.rope = rope;
  a.dtype = dtype;
  a.rope_base = rope_base;
  a.final_state = final_state;
  a.dbg_s = dbg_s;
  a.dbg_E = dbg_E;
  a.dbg_P = dbg_P;
  a.dbg_m = dbg_m;
  a.status = ws->status;
  a.ln = ln;
  a.ln_w = ln_w;
  a.ln_b = ln_b;
  a.ln_eps = ln_eps;
  if (rope && !use_chunk) {  // the chunked kernels compute their rotary factors themselves
    if (int rc = rope_table(ws, N, d, rope_base, st, &a.rope_table)) return rc;
  }
  if (use_chunk) {  // the scalar pass, then the chunked kernel
    const bool walk = walk_supported(d, dtype, causal) && !ln;
    const float* ang = nullptr;
    if (walk && rope) {
      if (int rc = walk_angles(ws, N, rope_base, st, &ang)) return rc;
    }
    void* buf = nullptr;
    const size_t scal_bytes = (size_t)B * H * N * sizeof(float4);
    const size_t smax_bytes = (size_t)B * H * kScalarCtas * sizeof(float);
    if (int rc = fwd_scratch(ws, scal_bytes + smax_bytes, &buf)) return rc;
    a.scal = static_cast<float4*>(buf);
    a.smax = reinterpret_cast<float*>(static_cast<char*>(buf) + scal_bytes);
    cudaError_t e = launch_fwd_scalars(a, a.scal, st);
    if (e != cudaSuccess) return cuda_fail(e, "forward scalar launch");
    e = walk ? launch_fwd_walk(a, ang, walk_max_segments(), st) : launch_fwd_chunk(a, st);
    if (e != cudaSuccess) return cuda_fail(e, "forward launch");
    return ZEROS_OK;
  }
  cudaError_t e = use_enc ? launch_fwd_encoder(a, st) : launch_fwd_simt(a, st);
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return ZEROS_OK;
}

int zeros_fwd_ex(const void* q, const void* k, const void* v, const void* u, const float* g1,
                 const float* gh, const float* g0, const float* mu, const float* tau, void* out,
                 int B, int H, int N, int d, int causal, int rope, int dtype, float rope_base,
                 int path, void* final_state, float* dbg_s, float* dbg_E, float* dbg_P,
                 float* dbg_m, void* stream) {
  return fwd_impl(q, k, v, u, g1, gh, g0, mu, tau, out, B, H, N, d, causal, rope, dtype,
                  rope_base, path, final_state, dbg_s, dbg_E, dbg_P, dbg_m, 0, nullptr, nullptr,
                  0.0f, stream);
}

int zeros_fwd_ln(const void* q, const void* k, const void* v, const void* u, const float* g1,
                 const float* gh, const float* g0, const float* mu, const float* tau,
                 const float* ln_w, const float* ln_b, float ln_eps, void* out, int B, int H,
                 int N, int d, int causal, int rope, int dtype, float rope_base, int path,
                 void* final_state, void* stream) {
  return fwd_impl(q, k, v, u, g1, gh, g0, mu, tau, out, B, H, N, d, causal, rope, dtype,
                  rope_base, path, final_state, nullptr, nullptr, nullptr, nullptr, 1, ln_w, ln_b,
                  ln_eps, stream);
}

int zeros_fwd(const void* q, const void* k, const void* v, const void* u, const float* g1,
              const float* gh, const float* mu, const float* tau, void* out, int B, int H, int N,
              int d, int causal, int rope, void* stream) {
  return zeros_fwd_ex(q, k, v, u, g1, gh, nullptr, mu, tau, out, B, H, N, d, causal, rope,
                      ZEROS_BF16,
                      10000.0f, ZEROS_PATH_AUTO, nullptr, nullptr, nullptr, nullptr, nullptr,
                      stream);
}

int zeros_fwd_noalloc(const void* q, const void* k, const void* v, const void* u,
                      const float* g1, const float* gh, const float* mu, const float* tau,
                      void* out, int B, int H, int N, int d, int causal, int rope, int dtype,
                      float rope_base, int* status, void* stream) {
  g_last_error.clear();
  if (int rc = check_dims(B, H, N, d)) return rc;
  if (int rc = check_dtype(dtype)) return rc;
  if (causal != 0 && causal != 1) return fail(ZEROS_ERR_INVALID, "causal must be 0 or 1");
  if (rope != 0 && rope != 1) return fail(ZEROS_ERR_INVALID, "rope must be 0 or 1");
  if (rope && !(rope_base > 0.0f)) return fail(ZEROS_ERR_INVALID, "rope_base must be > 0");
  const bool empty = (long long)B * H * N == 0;
  const char* names[] = {"q", "k", "v", "u", "g1", "gh", "mu", "tau", "out"};
  const void* ptrs[] = {q, k, v, u, g1, gh, mu, tau, out};
  if (!empty)
    for (int i = 0; i < 9; ++i)
      if (int rc = check_ptr(ptrs[i], names[i])) return rc;
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u))
    return fail(ZEROS_ERR_INVALID, "status is not 4-byte aligned");
  if (rope && (size_t)N * (size_t)(d / 2) > kNoAllocRopeEntries)
    return fail(ZEROS_ERR_UNSUPPORTED,
                "zeros_fwd_noalloc: N * d / 2 exceeds its fixed rotary scratch of 131072 entries");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (status) {
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), st);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
  }
  if (empty) return ZEROS_OK;
  FwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.u = u;
  a.g1 = g1;
  a.gh = gh;
  a.mu = mu;
  a.tau = tau;
  a.out = out;
  a.B = B;
  a.H = H;
  a.N = N;
  a.d = d;
  a.causal = causal;
  a.rope = rope;
  a.dtype = dtype;
  a.rope_base = rope_base;
  a.status = status;
  if (rope) {
    float2* table = nullptr;
    cudaError_t e = noalloc_rope_table(&table);
    if (e != cudaSuccess) return cuda_fail(e, "looking up the fixed rotary scratch");
    e = launch_rope_table(table, N, d, (double)rope_base, st);  // rewritten on every call
    if (e != cudaSuccess) return cuda_fail(e, "rotary table launch");
    a.rope_table = table;
  }
  cudaError_t e = launch_fwd_simt(a, st);
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return ZEROS_OK;
}

int zeros_state_init(void* state, const float* mu, const float* tau, int B, int H, int d,
                     int dtype, int rope, float rope_base, void* stream) {
  g_last_error.clear();
  if (int rc = check_dims(B, H, 0, d)) return rc;
  if (int rc = check_dtype(dtype)) return rc;
  if (rope != 0 && rope != 1) return fail(ZEROS_ERR_INVALID, "rope must be 0 or 1");
  if (rope && !(rope_base > 0.0f)) return fail(ZEROS_ERR_INVALID, "rope_base must be > 0");
  if (int rc = check_ptr(state, "state")) return rc;
  if ((long long)B * H > 0) {
    if (int rc = check_ptr(mu, "mu")) return rc;
    if (int rc = check_ptr(tau, "tau")) return rc;
  }
  DeviceWorkspace* ws;
  if (int rc = workspace(&ws)) return rc;
  cudaError_t e = launch_state_init(state, mu, tau, B, H, d, dtype, rope, rope_base,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "state init launch");
  std::lock_guard<std::mutex> lk(g_mutex);
  g_states[state] = StateInfo{B, H, d, dtype, rope, rope_base};
  return ZEROS_OK;
}

static int decode_impl(void* state, const StateInfo& si, const void* q, const void* k,
                       const void* v, const void* u, const float* g1, const float* gh,
                       const float* g0, void* out, float* dbg_s, float* dbg_E, float* dbg_P,
                       float* dbg_m, void* stream, int ln = 0, const float* ln_w = nullptr,
                       const float* ln_b = nullptr, float ln_eps = 0.0f) {
  if (int rc = check_dims(si.B, si.H, 1, si.d)) return rc;
  if (int rc = check_ln(ln, ln_w, ln_b, ln_eps)) return rc;
  if (int rc = check_ptr(state, "state")) return rc;
  if ((long long)si.B * si.H == 0) return ZEROS_OK;
  const char* names[] = {"q", "k", "v", "u", "g1", "gh", "out"};
  const void* ptrs[] = {q, k, v, u, g1, gh, out};
  for (int i = 0; i < 7; ++i)
    if (int rc = check_ptr(ptrs[i], names[i])) return rc;
  if (int rc = check_opt_ptr(g0, "g0")) return rc;
  if (int rc = check_opt_ptr(dbg_s, "dbg_s")) return rc;
  if (int rc = check_opt_ptr(dbg_E, "dbg_E")) return rc;
  if (int rc = check_opt_ptr(dbg_P, "dbg_P")) return rc;
  if (int rc = check_opt_ptr(dbg_m, "dbg_m")) return rc;
  DeviceWorkspace* ws;
  if (int rc = workspace(&ws)) return rc;
  DecodeArgs a{};
  a.state = state;
  a.q = q;
  a.k = k;
  a.v = v;
  a.u = u;
  a.g1 = g1;
  a.gh = gh;
  a.g0 = g0;
  a.out = out;
  a.B = si.B;
  a.H = si.H;
  a.d = si.d;
  a.dtype = si.dtype;
  a.rope = si.rope;
  a.rope_base = si.rope_base;
  a.dbg_s = dbg_s;
  a.dbg_E = dbg_E;
  a.dbg_P = dbg_P;
  a.dbg_m = dbg_m;
  a.status = ws->status;
  a.ln = ln;
  a.ln_w = ln_w;
  a.ln_b = ln_b;
  a.ln_eps = ln_eps;
  cudaError_t e = launch_decode(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return ZEROS_OK;
}

int zeros_decode_step(void* state, const void* q, const void* k, const void* v, const void* u,
                      const float* g1, const float* gh, void* out, void* stream) {
  g_last_error.clear();
  if (int rc = check_ptr(state, "state")) return rc;
  StateInfo si{};
  bool known = false;
  {
    std::lock_guard<std::mutex> lk(g_mutex);
    auto it = g_states.find(state);
    if (it != g_states.end()) {
      si = it->second;
      known = true;
    }
  }
  if (!known) {
    StateHeader hdr;
    cudaError_t e = cudaMemcpy(&hdr, state, sizeof(hdr), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the state header");
    if (std::memcmp(hdr.magic, "ZSP1", 4) != 0 || hdr.version != 1)
      return fail(ZEROS_ERR_INVALID, "state header not recognised");
    si = StateInfo{hdr.B, hdr.H, hdr.d, hdr.dtype, hdr.rope, hdr.rope_base};
    std::lock_guard<std::mutex> lk(g_mutex);
    g_states[state] = si;
  }
  return decode_impl(state, si, q, k, v, u, g1, gh, nullptr, out, nullptr, nullptr, nullptr,
                     nullptr, stream);
}

static int known_state(void* state, int B, int H, int d, StateInfo* out) {
  std::lock_guard<std::mutex> lk(g_mutex);
  auto it = g_states.find(state);
  if (it == g_states.end())
    return fail(ZEROS_ERR_INVALID,
                "state unknown to this process: create it with zeros_state_init or "
                "zeros_fwd_ex, or call zeros_decode_step once");
  if (it->second.B != B || it->second.H != H || it->second.d != d)
    return fail(ZEROS_ERR_INVALID, "dimensions differ from the state's");
  *out = it->second;
  return ZEROS_OK;
}

int zeros_decode_step_ln(void* state, int B, int H, int d, const void* q, const void* k,
                         const void* v, const void* u, const float* g1, const float* gh,
                         const float* g0, const float* ln_w, const float* ln_b, float ln_eps,
                         void* out, void* stream) {
  g_last_error.clear();
  StateInfo si{};
  if (int rc = known_state(state, B, H, d, &si)) return rc;
  return decode_impl(state, si, q, k, v, u, g1, gh, g0, out, nullptr, nullptr, nullptr, nullptr,
                     stream, 1, ln_w, ln_b, ln_eps);
}

int zeros_decode_step_ex(void* state, int B, int H, int d, const void* q, const void* k,
                         const void* v, const void* u, const float* g1, const float* gh,
                         const float* g0, void* out, float* dbg_s, float* dbg_E, float* dbg_P,
                         float* dbg_m, void* stream) {
  g_last_error.clear();
  StateInfo si{B, H, d, ZEROS_BF16, 0, 10000.0f};
  {
    std::lock_guard<std::mutex> lk(g_mutex);
    auto it = g_states.find(state);
    if (it != g_states.end()) {
      if (it->second.B != B || it->second.H != H || it->second.d != d)
        return fail(ZEROS_ERR_INVALID, "dimensions differ from the state's");
      si = it->second;
    } else {
      return fail(ZEROS_ERR_INVALID,
                  "state unknown to this process: create it with zeros_state_init or "
                  "zeros_fwd_ex, or call zeros_decode_step once");
    }
  }
  return decode_impl(state, si, q, k, v, u, g1, gh, g0, out, dbg_s, dbg_E, dbg_P, dbg_m,
                     stream);
}

int zeros_bwd_ex(const void* q, const void* k, const void* v, const void* u, const float* g1,
                 const float* gh, const float* g0, const float* mu, const float* tau,
                 const void* dout, float* dq, float* dk, float* dv, float* du, float* dg1,
                 float* dgh, float* dg0, float* dmu, float* dtau, int B, int H, int N, int d,
                 int rope, int dtype, float rope_base, int path, void* stream) {
  g_last_error.clear();
  if (int rc = check_dims(B, H, N, d)) return rc;
  if (path != ZEROS_PATH_AUTO && path != ZEROS_PATH_SIMT && path != ZEROS_PATH_CHUNK)
    return fail(ZEROS_ERR_INVALID, "unknown path");
  const unsigned long long n_chunks =
      (unsigned long long)B * H * (((unsigned long long)N + 63) / 64);
  const bool chunk_ok = bwd_chunk_supported(d) && n_chunks <= 0x7fffffffull;
  if (path == ZEROS_PATH_CHUNK && !chunk_ok)
    return fail(ZEROS_ERR_UNSUPPORTED, "the chunked backward needs d = 64");
  const bool use_chunk = chunk_ok && path != ZEROS_PATH_SIMT;
  if (int rc = check_dtype(dtype)) return rc;
  if (rope != 0 && rope != 1) return fail(ZEROS_ERR_INVALID, "rope must be 0 or 1");
  if (rope && !(rope_base > 0.0f)) return fail(ZEROS_ERR_INVALID, "rope_base must be > 0");
  if (dg0 && !g0) return fail(ZEROS_ERR_INVALID, "dg0 needs the zero-order gate g0");
  const char* names[] = {"q", "k", "v", "u", "g1", "gh", "dout", "dq", "dk", "dv", "du",
                         "dg1", "dgh"};
  const void* ptrs[] = {q, k, v, u, g1, gh, dout, dq, dk, dv, du, dg1, dgh};
  const bool empty = (long long)B * H * N == 0;
  if (!empty)
    for (int i = 0; i < 13; ++i)
      if (int rc = check_ptr(ptrs[i], names[i])) return rc;
  if (H > 0) {
    const char* n2[] = {"mu", "tau", "dmu", "dtau"};
    const void* p2[] = {mu, tau, dmu, dtau};
    for (int i = 0; i < 4; ++i)
      if (int rc = check_ptr(p2[i], n2[i])) return rc;
  }
  if (int rc = check_opt_ptr(g0, "g0")) return rc;
  if (int rc = check_opt_ptr(dg0, "dg0")) return rc;
  if (H == 0) return ZEROS_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // mu and tau gradients are sums over the batch: start from zero
  cudaError_t e = cudaMemsetAsync(dmu, 0, (size_t)H * d * sizeof(float), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(dtau, 0, (size_t)H * sizeof(float), st);
  if (e != cudaSuccess) return cuda_fail(e, "zeroing dmu / dtau");
  if (empty) return ZEROS_OK;
  DeviceWorkspace* ws;
  if (int rc = workspace(&ws)) return rc;
  BwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.u = u;
  a.dout = dout;
  a.g1 = g1;
  a.gh = gh;
  a.g0 = g0;
  a.mu = mu;
  a.tau = tau;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.du = du;
  a.dg1 = dg1;
  a.dgh = dgh;
  a.dg0 = dg0;
  a.dmu = dmu;
  a.dtau = dtau;
  a.B = B;
  a.H = H;
  a.N = N;
  a.d = d;
  a.rope = rope;
  a.dtype = dtype;
  a.status = ws->status;
  if (rope) {
    if (int rc = rope_table(ws, N, d, rope_base, st, &a.rope_table)) return rc;
  }
  if (!use_chunk) {
    if (int rc = bwd_scratch(ws, bwd_scratch_bytes(B, H, N, d), &a.scratch)) return rc;
    e = launch_bwd(a, st);
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    return ZEROS_OK;
  }
  // chunked: the forward's per-token scalars (the scalar pass for bf16 inputs, else a forward
  // launch whose output goes to scratch), then the state, chunk and scan kernels
  const size_t BHN = (size_t)B * H * N;
  const size_t out_bytes = ((BHN * d * (dtype == ZEROS_F32 ? 4 : 2)) + 255) / 256 * 256;
  float* buf = nullptr;
  if (int rc = bwd_scratch(ws, out_bytes + bwd_chunk_scratch_bytes(B, H, N, d), &buf)) return rc;
  float* scal = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(buf) + out_bytes);
  FwdArgs f{};
  f.q = q;
  f.k = k;
  f.v = v;
  f.u = u;
  f.g1 = g1;
  f.gh = gh;
  f.g0 = g0;
  f.mu = mu;
  f.tau = tau;
  f.out = buf;
  f.B = B;
  f.H = H;
  f.N = N;
  f.d = d;
  f.causal = 1;
  f.rope = rope;
  f.dtype = dtype;
  f.rope_base = rope_base;
  f.rope_table = a.rope_table;
  f.dbg_s = scal;
  f.dbg_E = scal + BHN;
  f.dbg_P = scal + 2 * BHN;
  f.dbg_m = scal + 3 * BHN;
  f.status = ws->status;
  if (chunk_supported(d, dtype, 1)) {
    static_assert(sizeof(float4) <= 64 * 2, "the scalars fit the forward output's scratch");
    e = launch_fwd_scalars(f, reinterpret_cast<float4*>(buf), st);
  } else {
    e = launch_fwd_simt(f, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "forward launch (backward scalars)");
  e = launch_bwd_chunk(a, scal, st);
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  return ZEROS_OK;
}

int zeros_bwd(const void* q, const void* k, const void* v, const void* u, const float* g1,
              const float* gh, const float* g0, const float* mu, const float* tau,
              const void* dout, float* dq, float* dk, float* dv, float* du, float* dg1,
              float* dgh, float* dg0, float* dmu, float* dtau, int B, int H, int N, int d,
              int rope, int dtype, float rope_base, void* stream) {
  return zeros_bwd_ex(q, k, v, u, g1, gh, g0, mu, tau, dout, dq, dk, dv, du, dg1, dgh, dg0, dmu,
                      dtau, B, H, N, d, rope, dtype, rope_base, ZEROS_PATH_AUTO, stream);
}

int zeros_sm_fwd(const void* q, const void* k, const void* v, const float* g1, const float* gh,
                 const float* g0, void* out, int B, int H, int N, int d, int causal, int rope,
                 int dtype, float rope_base, void* stream) {
  g_last_error.clear();
  if (int rc = check_dims(B, H, N, d)) return rc;
  if (int rc = check_dtype(dtype)) return rc;
  if (causal != 0 && causal != 1) return fail(ZEROS_ERR_INVALID, "causal must be 0 or 1");
  if (rope != 0 && rope != 1) return fail(ZEROS_ERR_INVALID, "rope must be 0 or 1");
  if (rope && !(rope_base > 0.0f)) return fail(ZEROS_ERR_INVALID, "rope_base must be > 0");
  if (!sm_supported(d, dtype))
    return fail(ZEROS_ERR_UNSUPPORTED, "ZeroS-SM needs bf16 inputs and d in {64, 128}");
  if (N > 65535 * 128) return fail(ZEROS_ERR_UNSUPPORTED, "ZeroS-SM needs N <= 8388480");
  const bool empty = (long long)B * H * N == 0;
  const char* names[] = {"q", "k", "v", "g1", "gh", "out"};
  const void* ptrs[] = {q, k, v, g1, gh, out};
  if (!empty)
    for (int i = 0; i < 6; ++i)
      if (int rc = check_ptr(ptrs[i], names[i])) return rc;
  if (int rc = check_opt_ptr(g0, "g0")) return rc;
  if (empty) return ZEROS_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DeviceWorkspace* ws;
  if (int rc = workspace(&ws)) return rc;
  SmArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.g1 = g1;
  a.gh = gh;
  a.g0 = g0;
  a.out = out;
  a.B = B;
  a.H = H;
  a.N = N;
  a.d = d;
  a.causal = causal;
  a.status = ws->status;
  // scratch: the rotated q and k (with rope), then (d = 64) the key-tile statistics
  const size_t each = rope ? (size_t)B * H * N * d * 2 : 0;
  const size_t ntiles = ((size_t)N + 127) / 128;
  const size_t stat_bytes = d == 64 ? (size_t)B * H * ntiles * kSmStat * sizeof(float) : 0;
  void* buf = nullptr;
  if (2 * each + stat_bytes > 0)
    if (int rc = sm_scratch(ws, 2 * each + stat_bytes, &buf)) return rc;
  const float2* table = nullptr;
  if (rope)
    if (int rc = rope_table(ws, N, d, rope_base, st, &table)) return rc;
  void* qr = buf;
  void* kr = static_cast<uint8_t*>(buf) + each;
  if (d == 64) {  // one pass: the statistics, and with rope the rotated q and k
    float* kstat = reinterpret_cast<float*>(static_cast<uint8_t*>(buf) + 2 * each);
    cudaError_t e = launch_sm_prep(q, k, v, qr, kr, rope ? table : nullptr, kstat, ws->status,
                                   B * H, N, st);
    if (e != cudaSuccess) return cuda_fail(e, "ZeroS-SM key statistics launch");
    a.kstat = kstat;
  } else if (rope) {
    cudaError_t e = launch_sm_rotate(q, k, qr, kr, table, B * H, N, d, st);
    if (e != cudaSuccess) return cuda_fail(e, "rotary launch");
  }
  if (rope) {
    a.q = qr;
    a.k = kr;
  }
  cudaError_t e = launch_sm(a, st);
  if (e != cudaSuccess) return cuda_fail(e, "ZeroS-SM launch");
  return ZEROS_OK;
}

int zeros_get_status(void* stream) {
  g_last_error.clear();
  DeviceWorkspace* ws;
  if (int rc = workspace(&ws)) return rc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int st = 0;
  e = cudaMemcpy(&st, ws->status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  if (st != 0) {
    e = cudaMemset(ws->status, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
  }
  return st;
}

}  // extern "C"
