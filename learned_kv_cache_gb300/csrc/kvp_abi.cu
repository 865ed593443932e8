// C ABI of libkvp: argument validation, dispatch to the kernels, status words.
//
// Every entry point validates its arguments on the host and returns an error
// before anything is enqueued; launches are asynchronous on the caller's
// stream; the library owns no memory except one int per device (the status
// word that kernels use to report device-side range errors and bounded-wait
// timeouts).
#include <algorithm>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>

#include "../../include/kvp.h"
#include "kvp_launch.h"

namespace {

thread_local std::string g_last_error;

__device__ int g_device_status;

constexpr int kMaxDevices = 64;
std::mutex g_status_mu;
int* g_status_ptr[kMaxDevices] = {nullptr};
void* g_status_ctx[kMaxDevices] = {nullptr};   // context each cached address belongs to

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(KVP_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Device address of this device's status word (looked up once per device and context).
int status_ptr(int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(KVP_ERR_UNSUPPORTED, "device ordinal %d", dev);
  void* ctx = kvp::current_cu_context();
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (!g_status_ptr[dev] || g_status_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_status);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
    g_status_ptr[dev] = (int*)p;
    g_status_ctx[dev] = ctx;
  }
  *out = g_status_ptr[dev];
  return KVP_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int elem_size(int dtype) { return dtype == KVP_F32 ? 4 : 2; }

int check_dtype(int dtype) {
  if (dtype != KVP_F32 && dtype != KVP_BF16 && dtype != KVP_F16)
    return fail(KVP_ERR_UNSUPPORTED, "dtype %d is not one of KVP_F32/KVP_BF16/KVP_F16", dtype);
  return KVP_OK;
}

int check_attn_shape(int n_batch, int h_q, int h_kv, int S, int D) {
  if (n_batch < 1 || h_q < 1 || h_kv < 1 || S < 1)
    return fail(KVP_ERR_INVALID_ARG, "n_batch=%d h_q=%d h_kv=%d seq_len=%d must be >= 1", n_batch,
                h_q, h_kv, S);
  if (h_q % h_kv != 0) return fail(KVP_ERR_INVALID_ARG, "h_q=%d not a multiple of h_kv=%d", h_q, h_kv);
  if (D != 64 && D != 128) return fail(KVP_ERR_UNSUPPORTED, "head_dim=%d (64 or 128 supported)", D);
  if ((long long)n_batch * h_q * S > (1LL << 40))
    return fail(KVP_ERR_INVALID_ARG, "problem too large");
  return KVP_OK;
}

// Shape and Q/K element strides of an attention pass.  strides == NULL means dense
// [n_batch, H, S, D]; otherwise {batch, head, token} strides in elements, each a positive
// multiple of 16 bytes (the head_dim axis is contiguous).  Strides of extent-1 dimensions are
// not used.
int attn_shape(int dtype, int n_batch, int h_q, int h_kv, int S, int D, const int64_t* q_strides,
               const int64_t* k_strides, kvp::AttnShape* out) {
  kvp::AttnShape s = kvp::dense_attn_shape(n_batch, h_q, h_kv, S, D);
  const int elt = elem_size(dtype);
  const int64_t* src[2] = {q_strides, k_strides};
  int64_t* dst[2] = {&s.q_sb, &s.k_sb};
  const char* name[2] = {"q_strides", "k_strides"};
  for (int t = 0; t < 2; ++t) {
    if (!src[t]) continue;
    for (int i = 0; i < 3; ++i) {
      const int64_t v = src[t][i];
      const bool used = i == 2 || (i == 0 ? n_batch > 1 : (t == 0 ? h_q : h_kv) > 1);
      if (!used) continue;
      if (v <= 0 || (v * elt) % 16 != 0 || v * elt >= (1LL << 40))
        return fail(KVP_ERR_INVALID_ARG,
                    "%s[%d]=%lld: strides must be positive multiples of 16 bytes below 2^40 bytes",
                    name[t], i, (long long)v);
      if (i == 2 && v < D)
        return fail(KVP_ERR_INVALID_ARG, "%s token stride %lld < head_dim %d", name[t], (long long)v, D);
    }
    dst[t][0] = n_batch > 1 ? src[t][0] : dst[t][0];
    dst[t][1] = (t == 0 ? h_q : h_kv) > 1 ? src[t][1] : dst[t][1];
    dst[t][2] = src[t][2];
  }
  *out = s;
  return KVP_OK;
}

// bf16 / f16 inputs run on the tensor-core passes, float32 inputs on the fp32-FFMA passes; there
// is no other path.  The tensor-core passes need the driver's tensor-map encoder.
int use_tensor_cores(int dtype, bool* tc) {
  *tc = dtype != KVP_F32;
  if (*tc && !kvp::tc_encoder_available())
    return fail(KVP_ERR_CUDA,
                "cuTensorMapEncodeTiled could not be resolved from the CUDA driver; bf16/f16 inputs "
                "run only on the tensor-core (TMA) passes");
  return KVP_OK;
}

std::atomic<unsigned long long> g_launches{0};

#define KVP_TRY(x)            \
  do {                        \
    int _rc = (x);            \
    if (_rc != KVP_OK) return _rc; \
  } while (0)

}  // namespace

namespace kvp {
void count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

void* current_cu_context() {
  typedef int (*CtxGetCurrentFn)(void**);
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  void* ctx = nullptr;
  if (fn && fn(&ctx) != 0) ctx = nullptr;
  return ctx;
}
}  // namespace kvp

extern "C" {

uint64_t kvp_launch_count(void) { return (uint64_t)g_launches.load(std::memory_order_relaxed); }

int kvp_abi_version(void) { return KVP_ABI_VERSION; }

const char* kvp_last_error(void) { return g_last_error.c_str(); }

const char* kvp_status_string(int status) {
  switch (status) {
    case KVP_OK: return "ok";
    case KVP_ERR_INVALID_ARG: return "invalid argument";
    case KVP_ERR_UNSUPPORTED: return "unsupported dtype, head_dim or layout";
    case KVP_ERR_CUDA: return "CUDA error";
    case KVP_ERR_TIMEOUT: return "bounded device wait timed out";
    case KVP_ERR_WORKSPACE: return "workspace missing or too small";
    case KVP_ERR_DEVICE_CHECK: return "device-side range check failed";
    default: return "unknown status";
  }
}

int kvp_check_device_status(kvp_stream_t stream) {
  int* st = nullptr;
  KVP_TRY(status_ptr(&st));
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol(status)");
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol(status)");
  if (v != KVP_OK) return fail(v, "device status: %s", kvp_status_string(v));
  return KVP_OK;
}

int kvp_lse_pass(const void* q, const void* k, int dtype, int n_batch, int h_q, int h_kv,
                 int seq_len, int head_dim, const int64_t* q_strides, const int64_t* k_strides,
                 float sm_scale, float* lse, kvp_stream_t stream) {
  g_last_error.clear();
  KVP_TRY(check_dtype(dtype));
  KVP_TRY(check_attn_shape(n_batch, h_q, h_kv, seq_len, head_dim));
  if (!q || !k || !lse) return fail(KVP_ERR_INVALID_ARG, "null q/k/lse");
  if (!aligned16(q) || !aligned16(k)) return fail(KVP_ERR_INVALID_ARG, "q/k not 16-byte aligned");
  if (!std::isfinite(sm_scale)) return fail(KVP_ERR_INVALID_ARG, "sm_scale not finite");
  kvp::AttnShape s;
  KVP_TRY(attn_shape(dtype, n_batch, h_q, h_kv, seq_len, head_dim, q_strides, k_strides, &s));
  bool tc = false;
  KVP_TRY(use_tensor_cores(dtype, &tc));
  int* st = nullptr;
  KVP_TRY(status_ptr(&st));
  cudaError_t e = tc ? kvp::launch_lse_tc(q, k, dtype, s, sm_scale, lse, st, (cudaStream_t)stream)
                     : kvp::launch_lse_simt(q, k, dtype, s, sm_scale, lse, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kvp_lse_pass launch");
  return KVP_OK;
}

int kvp_topk_cutoffs(const int32_t* ranks, int n_heads, int seq_len, int n_sink, int window, int k,
                     int32_t* tau, kvp_stream_t stream) {
  g_last_error.clear();
  if (!ranks || !tau) return fail(KVP_ERR_INVALID_ARG, "null ranks/tau");
  if (n_heads < 1 || n_heads > 65535) return fail(KVP_ERR_INVALID_ARG, "n_heads=%d", n_heads);
  if (seq_len < 1 || seq_len > (1 << 19)) return fail(KVP_ERR_INVALID_ARG, "seq_len=%d", seq_len);
  if (k < 1) return fail(KVP_ERR_INVALID_ARG, "k=%d must be >= 1", k);
  if (n_sink < 0 || window < 0) return fail(KVP_ERR_INVALID_ARG, "n_sink=%d window=%d", n_sink, window);
  int* st = nullptr;
  KVP_TRY(status_ptr(&st));
  cudaError_t e = kvp::launch_topk_cutoffs(ranks, n_heads, seq_len, n_sink, window, k, tau, st,
                                           (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kvp_topk_cutoffs launch");
  return KVP_OK;
}

size_t kvp_sparse_lse_workspace_size(int dtype, int n_batch, int h_q, int h_kv, int seq_len, int head_dim) {
  if (check_dtype(dtype) != KVP_OK || check_attn_shape(n_batch, h_q, h_kv, seq_len, head_dim) != KVP_OK)
    return 0;
  return kvp::sparse_lse_workspace_size(dtype, kvp::dense_attn_shape(n_batch, h_q, h_kv, seq_len, head_dim));
}

int kvp_sparse_lse_pass(const void* q, const void* k, const int32_t* ranks, const int32_t* tau,
                        int dtype, int n_batch, int h_q, int h_kv, int seq_len, int head_dim,
                        const int64_t* q_strides, const int64_t* k_strides, float sm_scale,
                        int n_sink, int window, float* lse, void* workspace, size_t workspace_bytes,
                        kvp_stream_t stream) {
  g_last_error.clear();
  KVP_TRY(check_dtype(dtype));
  KVP_TRY(check_attn_shape(n_batch, h_q, h_kv, seq_len, head_dim));
  if (!q || !k || !lse || !ranks || !tau) return fail(KVP_ERR_INVALID_ARG, "null q/k/ranks/tau/lse");
  if (!aligned16(q) || !aligned16(k)) return fail(KVP_ERR_INVALID_ARG, "q/k not 16-byte aligned");
  if (!std::isfinite(sm_scale)) return fail(KVP_ERR_INVALID_ARG, "sm_scale not finite");
  if (n_sink < 0 || window < 0) return fail(KVP_ERR_INVALID_ARG, "n_sink=%d window=%d", n_sink, window);
  kvp::AttnShape s;
  KVP_TRY(attn_shape(dtype, n_batch, h_q, h_kv, seq_len, head_dim, q_strides, k_strides, &s));
  bool tc = false;
  KVP_TRY(use_tensor_cores(dtype, &tc));
  int* st = nullptr;
  KVP_TRY(status_ptr(&st));
  kvp::SparseMask mask{ranks, tau, n_sink, window};
  const size_t need = kvp::sparse_lse_workspace_size(dtype, s);
  if (need > 0) {
    if (!workspace || workspace_bytes < need)
      return fail(KVP_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
    if (((uintptr_t)workspace & 255) != 0) return fail(KVP_ERR_INVALID_ARG, "workspace not 256-byte aligned");
    const size_t n = (size_t)n_batch * h_kv * seq_len;
    const size_t inv_bytes = (n * 4 + 255) & ~(size_t)255;
    const size_t ks_bytes = (n * (size_t)head_dim * 2 + 255) & ~(size_t)255;
    char* w = (char*)workspace;
    mask.inv = (int32_t*)w;
    mask.k_sorted = w + inv_bytes;
    mask.perm_ok = (int*)(w + inv_bytes + ks_bytes);
  }
  cudaError_t e = tc ? kvp::launch_lse_tc(q, k, dtype, s, sm_scale, lse, st, (cudaStream_t)stream, &mask)
                     : kvp::launch_lse_simt(q, k, dtype, s, sm_scale, lse, (cudaStream_t)stream, &mask);
  if (e != cudaSuccess) return cuda_fail(e, "kvp_sparse_lse_pass launch");
  return KVP_OK;
}

size_t kvp_future_attn_mass_workspace_size(int dtype, int n_batch, int h_q, int h_kv, int seq_len,
                                           int head_dim, int window) {
  if (check_dtype(dtype) != KVP_OK || check_attn_shape(n_batch, h_q, h_kv, seq_len, head_dim) != KVP_OK ||
      window < 0)
    return 0;
  const kvp::AttnShape s = kvp::dense_attn_shape(n_batch, h_q, h_kv, seq_len, head_dim);
  return dtype != KVP_F32 ? kvp::fam_tc_workspace_size(s, window) : 0;
}

int kvp_future_attn_mass(const void* q, const void* k, const float* lse, int dtype, int n_batch,
                         int h_q, int h_kv, int seq_len, int head_dim, const int64_t* q_strides,
                         const int64_t* k_strides, float sm_scale, int window, float* F,
                         void* workspace, size_t workspace_bytes, kvp_stream_t stream) {
  g_last_error.clear();
  KVP_TRY(check_dtype(dtype));
  KVP_TRY(check_attn_shape(n_batch, h_q, h_kv, seq_len, head_dim));
  if (!q || !k || !lse || !F) return fail(KVP_ERR_INVALID_ARG, "null q/k/lse/F");
  if (!aligned16(q) || !aligned16(k)) return fail(KVP_ERR_INVALID_ARG, "q/k not 16-byte aligned");
  if (window < 0) return fail(KVP_ERR_INVALID_ARG, "window=%d < 0", window);
  if (!std::isfinite(sm_scale)) return fail(KVP_ERR_INVALID_ARG, "sm_scale not finite");
  kvp::AttnShape s;
  KVP_TRY(attn_shape(dtype, n_batch, h_q, h_kv, seq_len, head_dim, q_strides, k_strides, &s));
  bool tc = false;
  KVP_TRY(use_tensor_cores(dtype, &tc));
  const size_t need = kvp_future_attn_mass_workspace_size(dtype, n_batch, h_q, h_kv, seq_len,
                                                          head_dim, window);
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(KVP_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  int* st = nullptr;
  KVP_TRY(status_ptr(&st));
  cudaError_t e = tc ? kvp::launch_fam_tc(q, k, lse, dtype, s, sm_scale, window, F, workspace,
                                          workspace_bytes, st, (cudaStream_t)stream)
                     : kvp::launch_fam_simt(q, k, lse, dtype, s, sm_scale, window, F, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kvp_future_attn_mass launch");
  return KVP_OK;
}

static size_t target_heads_bytes(int n_batch, int h_q, int seq_len) {
  return (((size_t)n_batch * h_q * seq_len * sizeof(float)) + 255) & ~(size_t)255;
}

size_t kvp_future_attn_target_workspace_size(int dtype, int n_batch, int h_q, int h_kv, int seq_len,
                                             int head_dim, int window) {
  if (check_dtype(dtype) != KVP_OK || check_attn_shape(n_batch, h_q, h_kv, seq_len, head_dim) != KVP_OK ||
      window < 0)
    return 0;
  const kvp::AttnShape s = kvp::dense_attn_shape(n_batch, h_q, h_kv, seq_len, head_dim);
  const size_t part = dtype != KVP_F32 ? kvp::fam_tc_workspace_size(s, window, 1) : 0;
  return target_heads_bytes(n_batch, h_q, seq_len) + part;
}

int kvp_future_attn_target(const void* q, const void* k, const float* lse, int dtype, int n_batch,
                           int h_q, int h_kv, int seq_len, int head_dim, const int64_t* q_strides,
                           const int64_t* k_strides, float sm_scale, int window, float eps,
                           int aggregate, float* target, float* F_heads, float* F, void* workspace,
                           size_t workspace_bytes, kvp_stream_t stream) {
  g_last_error.clear();
  KVP_TRY(check_dtype(dtype));
  KVP_TRY(check_attn_shape(n_batch, h_q, h_kv, seq_len, head_dim));
  if (!q || !k || !lse) return fail(KVP_ERR_INVALID_ARG, "null q/k/lse");
  if (!target && !F_heads && !F) return fail(KVP_ERR_INVALID_ARG, "no output requested");
  if (!aligned16(q) || !aligned16(k)) return fail(KVP_ERR_INVALID_ARG, "q/k not 16-byte aligned");
  if (window < 0) return fail(KVP_ERR_INVALID_ARG, "window=%d < 0", window);
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return fail(KVP_ERR_INVALID_ARG, "sm_scale must be > 0");
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(KVP_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (aggregate != KVP_TARGET_MAX_LOG && aggregate != KVP_TARGET_MEAN_PROB)
    return fail(KVP_ERR_INVALID_ARG, "aggregate=%d", aggregate);
  kvp::AttnShape s;
  KVP_TRY(attn_shape(dtype, n_batch, h_q, h_kv, seq_len, head_dim, q_strides, k_strides, &s));
  bool tc = false;
  KVP_TRY(use_tensor_cores(dtype, &tc));
  const size_t need = kvp_future_attn_target_workspace_size(dtype, n_batch, h_q, h_kv, seq_len, head_dim, window);
  if (!workspace || workspace_bytes < need)
    return fail(KVP_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  if (((uintptr_t)workspace & 255u) != 0) return fail(KVP_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  int* st = nullptr;
  KVP_TRY(status_ptr(&st));
  char* part = (char*)workspace + target_heads_bytes(n_batch, h_q, seq_len);
  if (tc) {
    // the per-head sums go straight into the target (and F_heads / F when asked for)
    const kvp::TargetOut to{eps, aggregate, target, F};
    cudaError_t e = kvp::launch_fam_tc(q, k, lse, dtype, s, sm_scale, window, F_heads, part,
                                       workspace_bytes - target_heads_bytes(n_batch, h_q, seq_len), st,
                                       (cudaStream_t)stream, 1, &to);
    if (e != cudaSuccess) return cuda_fail(e, "kvp_future_attn_target launch");
    return KVP_OK;
  }
  float* heads = F_heads ? F_heads : (float*)workspace;
  cudaError_t e = kvp::launch_fam_simt(q, k, lse, dtype, s, sm_scale, window, heads, (cudaStream_t)stream, 1);
  if (e != cudaSuccess) return cuda_fail(e, "kvp_future_attn_target launch");
  if (target || F) {
    e = kvp::launch_target_epilogue(heads, n_batch, h_q, h_kv, seq_len, window, eps, aggregate, target, F,
                                    (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "kvp_future_attn_target epilogue");
  }
  return KVP_OK;
}

int kvp_soft_topk_budgets(const double* scores, int n, double k, int t, double* ratios,
                          int32_t* budgets, kvp_stream_t stream) {
  g_last_error.clear();
  if (!scores || !ratios || !budgets) return fail(KVP_ERR_INVALID_ARG, "null scores/ratios/budgets");
  if (n < 1 || n > 1024) return fail(KVP_ERR_INVALID_ARG, "n=%d outside [1, 1024]", n);
  if (!(k > 0.0 && k < (double)n)) return fail(KVP_ERR_INVALID_ARG, "k=%g outside (0, n)", k);
  if (t < 0) return fail(KVP_ERR_INVALID_ARG, "t=%d < 0", t);
  cudaError_t e = kvp::launch_soft_topk(scores, n, k, t, ratios, budgets, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kvp_soft_topk_budgets launch");
  return KVP_OK;
}

int kvp_select_topk(const float* scores, int R, int T, int64_t row_stride, const int32_t* budgets,
                    int n_sink, int n_recent, int32_t* idx, int b_max, int32_t* count,
                    kvp_stream_t stream) {
  g_last_error.clear();
  if (!scores || !budgets || !idx || !count) return fail(KVP_ERR_INVALID_ARG, "null pointer");
  if (R < 1 || T < 1) return fail(KVP_ERR_INVALID_ARG, "R=%d T=%d must be >= 1", R, T);
  if (row_stride < T) return fail(KVP_ERR_INVALID_ARG, "row_stride=%lld < T=%d", (long long)row_stride, T);
  if (n_sink < 0 || n_recent < 0) return fail(KVP_ERR_INVALID_ARG, "negative n_sink/n_recent");
  if (b_max < 1) return fail(KVP_ERR_INVALID_ARG, "b_max=%d must be >= 1", b_max);
  if (R > 2147483647 / 2) return fail(KVP_ERR_INVALID_ARG, "R too large");
  int* st = nullptr;
  KVP_TRY(status_ptr(&st));
  cudaError_t e = kvp::launch_select(scores, R, T, row_stride, budgets, n_sink, n_recent, idx, b_max,
                                     count, st, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kvp_select_topk launch");
  return KVP_OK;
}

int kvp_compact_kv(const void* k, const void* v, int dtype, int R, int T, int head_dim,
                   const int32_t* idx, const int32_t* count, int b_max, void* k_out, void* v_out,
                   kvp_stream_t stream) {
  g_last_error.clear();
  KVP_TRY(check_dtype(dtype));
  if (!k || !v || !idx || !count || !k_out || !v_out) return fail(KVP_ERR_INVALID_ARG, "null pointer");
  if (R < 1 || T < 1 || b_max < 1) return fail(KVP_ERR_INVALID_ARG, "R=%d T=%d b_max=%d must be >= 1", R, T, b_max);
  if (head_dim != 64 && head_dim != 128) return fail(KVP_ERR_UNSUPPORTED, "head_dim=%d", head_dim);
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_out) || !aligned16(v_out))
    return fail(KVP_ERR_INVALID_ARG, "k/v/k_out/v_out not 16-byte aligned");
  int* st = nullptr;
  KVP_TRY(status_ptr(&st));
  cudaError_t e = kvp::launch_compact(k, v, head_dim * elem_size(dtype), R, T, idx, count, b_max,
                                      k_out, v_out, st, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kvp_compact_kv launch");
  return KVP_OK;
}

int kvp_chunk_compress(const void* cache_k, const void* cache_v, const float* cache_score,
                       const int32_t* cache_pos, int cap_in, int n_in, const void* chunk_k,
                       const void* chunk_v, const float* chunk_score, int chunk_len, int pos0,
                       int dtype, int R, int head_dim, int budget, int n_sink, int n_recent,
                       int32_t* idx, int32_t* count, void* out_k, void* out_v, float* out_score,
                       int32_t* out_pos, int out_cap, kvp_stream_t stream) {
  g_last_error.clear();
  KVP_TRY(check_dtype(dtype));
  if (!chunk_k || !chunk_v || !chunk_score || !idx || !count || !out_k || !out_v || !out_score || !out_pos)
    return fail(KVP_ERR_INVALID_ARG, "null pointer");
  if (n_in > 0 && (!cache_k || !cache_v || !cache_score || !cache_pos))
    return fail(KVP_ERR_INVALID_ARG, "null cache pointer with n_in=%d", n_in);
  if (R < 1 || chunk_len < 1 || n_in < 0 || n_in > cap_in)
    return fail(KVP_ERR_INVALID_ARG, "R=%d chunk_len=%d n_in=%d cap_in=%d", R, chunk_len, n_in, cap_in);
  if ((long long)n_in + chunk_len > 0x7fffffffLL) return fail(KVP_ERR_INVALID_ARG, "n_in + chunk_len overflows");
  if (head_dim != 64 && head_dim != 128) return fail(KVP_ERR_UNSUPPORTED, "head_dim=%d", head_dim);
  if (budget < 1 || n_sink < 0 || n_recent < 0)
    return fail(KVP_ERR_INVALID_ARG, "budget=%d n_sink=%d n_recent=%d", budget, n_sink, n_recent);
  if (pos0 < 0) return fail(KVP_ERR_INVALID_ARG, "pos0=%d < 0", pos0);
  const int T = n_in + chunk_len;
  const int b_eff = T <= budget ? T : std::min(T, std::max(budget, n_sink + n_recent));
  if (out_cap < b_eff) return fail(KVP_ERR_INVALID_ARG, "out_cap=%d < kept count %d", out_cap, b_eff);
  if ((n_in > 0 && (!aligned16(cache_k) || !aligned16(cache_v))) || !aligned16(chunk_k) ||
      !aligned16(chunk_v) || !aligned16(out_k) || !aligned16(out_v))
    return fail(KVP_ERR_INVALID_ARG, "K/V buffers not 16-byte aligned");
  int* st = nullptr;
  KVP_TRY(status_ptr(&st));
  cudaError_t e = kvp::launch_select(n_in > 0 ? cache_score : chunk_score, R, T,
                                     n_in > 0 ? (int64_t)cap_in : (int64_t)chunk_len, nullptr, n_sink,
                                     n_recent, idx, out_cap, count, st, (cudaStream_t)stream,
                                     n_in > 0 ? chunk_score : nullptr, chunk_len, n_in, budget);
  if (e != cudaSuccess) return cuda_fail(e, "kvp_chunk_compress select launch");
  const kvp::ChunkSrc src{cache_k, cache_v, cache_score, cache_pos, cap_in, n_in,
                          chunk_k, chunk_v, chunk_score, chunk_len, pos0};
  e = kvp::launch_chunk_compact(src, head_dim * elem_size(dtype), R, idx, count, out_cap, out_k, out_v,
                                out_score, out_pos, out_cap, st, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kvp_chunk_compress compact launch");
  return KVP_OK;
}

size_t kvp_rank_rows_workspace_size(int R, int T) {
  if (R < 1 || R > 65535 || T < 1) return 0;
  return kvp::rank_rows_workspace_size(R, T);
}

int kvp_rank_rows(const float* scores, int R, int T, int32_t* ranks, void* workspace,
                  size_t workspace_bytes, kvp_stream_t stream) {
  g_last_error.clear();
  if (!scores || !ranks) return fail(KVP_ERR_INVALID_ARG, "null scores/ranks");
  if (R < 1 || R > 65535 || T < 1) return fail(KVP_ERR_INVALID_ARG, "R=%d T=%d", R, T);
  const size_t need = kvp::rank_rows_workspace_size(R, T);
  if (!workspace || workspace_bytes < need)
    return fail(KVP_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  if (((uintptr_t)workspace & 255) != 0) return fail(KVP_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  int* st = nullptr;
  KVP_TRY(status_ptr(&st));
  cudaError_t e = kvp::launch_rank_rows(scores, R, T, ranks, workspace, st, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kvp_rank_rows launch");
  return KVP_OK;
}

size_t kvp_eviction_auc_workspace_size(int R, int M, int T) {
  if (R < 1 || R > 65535 || M < 1 || M > 65535 || (long long)R * M > (1LL << 24) || T < 1) return 0;
  return kvp::eviction_auc_workspace_size(R, M, T);
}

int kvp_eviction_auc(const float* F, const int32_t* ranks, int R, int M, int T, double* auc,
                     void* workspace, size_t workspace_bytes, kvp_stream_t stream) {
  g_last_error.clear();
  if (!F || !ranks || !auc) return fail(KVP_ERR_INVALID_ARG, "null F/ranks/auc");
  if (R < 1 || R > 65535 || M < 1 || M > 65535 || (long long)R * M > (1LL << 24) || T < 1)
    return fail(KVP_ERR_INVALID_ARG, "R=%d M=%d T=%d", R, M, T);
  const size_t need = kvp::eviction_auc_workspace_size(R, M, T);
  if (!workspace || workspace_bytes < need)
    return fail(KVP_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  if (((uintptr_t)workspace & 7) != 0) return fail(KVP_ERR_INVALID_ARG, "workspace not 8-byte aligned");
  cudaError_t e = kvp::launch_eviction_auc(F, ranks, R, M, T, auc, workspace, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kvp_eviction_auc launch");
  return KVP_OK;
}

int kvp_ring_insert(void* kc, void* vc, int32_t* slot_pos, float* slot_score, int32_t* fill,
                    int dtype, int R, int cap, int head_dim, const void* new_k, const void* new_v,
                    int new_pos, int n_sink, int n_recent, int32_t* out_slot, kvp_stream_t stream) {
  g_last_error.clear();
  KVP_TRY(check_dtype(dtype));
  if (!kc || !vc || !slot_pos || !slot_score || !fill || !new_k || !new_v)
    return fail(KVP_ERR_INVALID_ARG, "null pointer");
  if (R < 1 || cap < 1) return fail(KVP_ERR_INVALID_ARG, "R=%d cap=%d must be >= 1", R, cap);
  if (head_dim != 64 && head_dim != 128) return fail(KVP_ERR_UNSUPPORTED, "head_dim=%d", head_dim);
  if (n_sink < 0 || n_recent < 1) return fail(KVP_ERR_INVALID_ARG, "need n_sink >= 0 and n_recent >= 1");
  if (cap < n_sink + n_recent)
    return fail(KVP_ERR_INVALID_ARG, "cap=%d < n_sink + n_recent = %d: a full cache would have nothing to evict",
                cap, n_sink + n_recent);
  if (new_pos < 0) return fail(KVP_ERR_INVALID_ARG, "new_pos=%d < 0", new_pos);
  if (!aligned16(kc) || !aligned16(vc) || !aligned16(new_k) || !aligned16(new_v))
    return fail(KVP_ERR_INVALID_ARG, "kc/vc/new_k/new_v not 16-byte aligned");
  int* st = nullptr;
  KVP_TRY(status_ptr(&st));
  cudaError_t e = kvp::launch_ring_insert(kc, vc, slot_pos, slot_score, fill, R, cap, head_dim * elem_size(dtype),
                                          new_k, new_v, new_pos, n_sink, n_recent, out_slot, st,
                                          (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kvp_ring_insert launch");
  return KVP_OK;
}

size_t kvp_decode_attn_workspace_size(int n_layers, int h_q, int h_kv, int head_dim, int T_cap,
                                      int with_key_mass) {
  if (n_layers < 1 || h_q < 1 || h_kv < 1 || h_q % h_kv || T_cap < 1 ||
      (head_dim != 64 && head_dim != 128))
    return 0;
  return kvp::decode_plan(n_layers, h_q, h_kv, head_dim, T_cap, with_key_mass).total_bytes;
}

int kvp_decode_attn(const void* q, const void* kc, const void* vc, int dtype, int n_layers, int h_q,
                    int h_kv, int head_dim, int T_cap, const int32_t* len, float sm_scale,
                    float* out, float* key_mass, const int32_t* key_pos, int T_src, int accumulate,
                    void* workspace, size_t workspace_bytes, kvp_stream_t stream) {
  g_last_error.clear();
  KVP_TRY(check_dtype(dtype));
  if (!q || !kc || !vc || !len || !out) return fail(KVP_ERR_INVALID_ARG, "null q/kc/vc/len/out");
  if (n_layers < 1 || h_q < 1 || h_kv < 1 || T_cap < 1)
    return fail(KVP_ERR_INVALID_ARG, "n_layers=%d h_q=%d h_kv=%d T_cap=%d must be >= 1", n_layers,
                h_q, h_kv, T_cap);
  if (h_q % h_kv) return fail(KVP_ERR_INVALID_ARG, "h_q=%d not a multiple of h_kv=%d", h_q, h_kv);
  if (h_q / h_kv > 8) return fail(KVP_ERR_UNSUPPORTED, "group size %d > 8", h_q / h_kv);
  if (head_dim != 64 && head_dim != 128) return fail(KVP_ERR_UNSUPPORTED, "head_dim=%d", head_dim);
  if (!aligned16(q) || !aligned16(kc) || !aligned16(vc))
    return fail(KVP_ERR_INVALID_ARG, "q/kc/vc not 16-byte aligned");
  if (!std::isfinite(sm_scale)) return fail(KVP_ERR_INVALID_ARG, "sm_scale not finite");
  if (key_mass) {
    if (T_src < 1) return fail(KVP_ERR_INVALID_ARG, "T_src=%d must be >= 1", T_src);
    if (!key_pos && T_src < T_cap)
      return fail(KVP_ERR_INVALID_ARG, "T_src=%d < T_cap=%d without key_pos", T_src, T_cap);
    if (accumulate != 0 && accumulate != 1) return fail(KVP_ERR_INVALID_ARG, "accumulate must be 0 or 1");
  }
  const kvp::DecodePlan plan = kvp::decode_plan(n_layers, h_q, h_kv, head_dim, T_cap, key_mass != nullptr);
  if (!workspace || workspace_bytes < plan.total_bytes)
    return fail(KVP_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", plan.total_bytes,
                workspace_bytes);
  if (((uintptr_t)workspace & 255u) != 0) return fail(KVP_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  int* st = nullptr;
  KVP_TRY(status_ptr(&st));
  cudaError_t e = kvp::launch_decode(q, kc, vc, dtype, n_layers, h_q, h_kv, head_dim, T_cap, len,
                                     sm_scale, out, key_mass, key_pos, T_src, accumulate, plan,
                                     workspace, st, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kvp_decode_attn launch");
  return KVP_OK;
}

int kvp_decode_attn_noalloc(const void* q, const void* kc, const void* vc, int dtype, int n_layers,
                            int h_q, int h_kv, int head_dim, int T_cap, const int32_t* len,
                            float sm_scale, float* out, kvp_stream_t stream) {
  g_last_error.clear();
  KVP_TRY(check_dtype(dtype));
  if (!q || !kc || !vc || !len || !out) return fail(KVP_ERR_INVALID_ARG, "null q/kc/vc/len/out");
  if (n_layers < 1 || h_q < 1 || h_kv < 1 || T_cap < 1)
    return fail(KVP_ERR_INVALID_ARG, "n_layers=%d h_q=%d h_kv=%d T_cap=%d must be >= 1", n_layers,
                h_q, h_kv, T_cap);
  if (h_q % h_kv) return fail(KVP_ERR_INVALID_ARG, "h_q=%d not a multiple of h_kv=%d", h_q, h_kv);
  if (h_q / h_kv > 8) return fail(KVP_ERR_UNSUPPORTED, "group size %d > 8", h_q / h_kv);
  if (head_dim != 64 && head_dim != 128) return fail(KVP_ERR_UNSUPPORTED, "head_dim=%d", head_dim);
  if (!aligned16(q) || !aligned16(kc) || !aligned16(vc))
    return fail(KVP_ERR_INVALID_ARG, "q/kc/vc not 16-byte aligned");
  if (!std::isfinite(sm_scale)) return fail(KVP_ERR_INVALID_ARG, "sm_scale not finite");
  const kvp::DecodePlan plan = kvp::decode_plan(n_layers, h_q, h_kv, head_dim, T_cap, 0);
  if (plan.total_bytes > (size_t)KVP_DECODE_NOALLOC_SCRATCH_BYTES)
    return fail(KVP_ERR_WORKSPACE,
                "this shape needs %zu bytes of scratch; the built-in scratch of "
                "kvp_decode_attn_noalloc holds %zu (use kvp_decode_attn with a workspace)",
                plan.total_bytes, (size_t)KVP_DECODE_NOALLOC_SCRATCH_BYTES);
  if (!kvp::decode_noalloc_scratch_ready()) {
    // The first call on a device (and context) looks up the scratch address, which a stream
    // capture does not allow: ask for an uncaptured first call instead.
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t ce = cudaStreamIsCapturing((cudaStream_t)stream, &cs);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamIsCapturing");
    if (cs != cudaStreamCaptureStatusNone)
      return fail(KVP_ERR_INVALID_ARG,
                  "kvp_decode_attn_noalloc: the first call on this device sets up its scratch address "
                  "and cannot run under stream capture; make one call before capturing");
  }
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  cudaError_t e = kvp::decode_noalloc_scratch(&scratch, &scratch_bytes);
  if (e != cudaSuccess) return cuda_fail(e, "kvp_decode_attn_noalloc scratch lookup");
  if (scratch_bytes < plan.total_bytes) return fail(KVP_ERR_WORKSPACE, "scratch smaller than plan");
  int* st = nullptr;
  KVP_TRY(status_ptr(&st));
  e = kvp::launch_decode(q, kc, vc, dtype, n_layers, h_q, h_kv, head_dim, T_cap, len, sm_scale, out,
                         nullptr, nullptr, 0, 0, plan, scratch, st, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kvp_decode_attn_noalloc launch");
  return KVP_OK;
}

}  // extern "C"
