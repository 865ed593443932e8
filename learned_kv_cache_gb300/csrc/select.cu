// Budgeted selection (sinks + recent window + top-k) and Soft-TopK head budgets.
//
// Selection (KVpop "The KVpop Scoring Module"; Learning to Evict from
// Key-Value Cache §A.2; How much KV cache can you prune "What we did"):
// one CTA per row.  Scores are mapped to order-preserving uint32 keys (NaN
// lowest, -0.0 folded onto +0.0); a 4-pass 8-bit radix select finds the k-th
// largest key v* and how many of the keys equal to v* must be kept; a final
// pass in token order keeps keys > v*, the first `remaining` keys == v*
// (lowest indices first) and the sinks / recent window, and writes their
// indices in ascending order through a block-wide prefix scan.
//
// Soft-TopK (LKV "The Differentiable Soft-TopK Operator", "LKV-H"): one CTA
// sorts the n <= 1024 head scores, forms the prefix sums S1 = sum exp(-x) and
// suffix sums S2 = sum exp(x), evaluates the closed-form threshold for every
// split m and keeps the split that is consistent (top m scores at or above
// the threshold); ratios are the Laplace CDF of (x - lambda), b = floor(r*t).
#include <float.h>

#include "kvp_common.cuh"
#include "kvp_launch.h"

namespace kvp {
namespace {

__device__ __forceinline__ uint32_t order_key(float x) {
  if (x != x) return 0u;                  // NaN ranks below every number
  uint32_t u = __float_as_uint(x);
  if ((u << 1) == 0u) u = 0u;             // -0.0 == +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int SEL_THREADS = 1024;
constexpr int SEL_ITEMS = 4;              // consecutive tokens per thread in the output pass

__global__ void __launch_bounds__(SEL_THREADS) select_kernel(
    const float* __restrict__ scores, int T, long long row_stride, const int32_t* __restrict__ budgets,
    int n_sink, int n_recent, int32_t* __restrict__ idx, int b_max, int32_t* __restrict__ count,
    int* status) {
  __shared__ int hist[256];
  __shared__ int scan_sh[33];
  __shared__ int sel_digit, sel_remaining;
  const int r = blockIdx.x;
  const float* s = scores + (size_t)r * row_stride;
  int32_t* out = idx + (size_t)r * b_max;
  const int b = budgets[r];
  if (b < 0) {
    if (threadIdx.x == 0) { count[r] = -1; raise_status(status, KVP_ERR_DEVICE_CHECK); }
    return;
  }
  const int b_eff = (T <= b) ? T : min(T, max(b, n_sink + n_recent));
  if (b_eff > b_max) {
    if (threadIdx.x == 0) { count[r] = -1; raise_status(status, KVP_ERR_DEVICE_CHECK); }
    return;
  }
  const bool keep_all = b_eff >= T;
  const int mid_lo = n_sink, mid_hi = T - n_recent;
  int k = keep_all ? 0 : b_eff - n_sink - n_recent;

  uint32_t prefix = 0u, mask = 0u;
  int remaining = k;
  if (k > 0) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      for (int i = mid_lo + threadIdx.x; i < mid_hi; i += blockDim.x) {
        const uint32_t key = order_key(s[i]);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        int cum = 0, d = 255;
        for (; d > 0; --d) {
          if (cum + hist[d] >= remaining) break;
          cum += hist[d];
        }
        sel_digit = d;
        sel_remaining = remaining - cum;
      }
      __syncthreads();
      prefix |= (uint32_t)sel_digit << shift;
      mask |= 255u << shift;
      remaining = sel_remaining;
      __syncthreads();
    }
  }
  const uint32_t vstar = prefix;
  // Output pass in token order.
  int base = 0, eq_base = 0;
  for (int c0 = 0; c0 < T; c0 += SEL_THREADS * SEL_ITEMS) {
    const int i_first = c0 + threadIdx.x * SEL_ITEMS;
    uint32_t keys[SEL_ITEMS];
    int n_eq = 0;
#pragma unroll
    for (int t = 0; t < SEL_ITEMS; ++t) {
      const int i = i_first + t;
      keys[t] = 0u;
      if (k > 0 && i < T && i >= mid_lo && i < mid_hi) {
        keys[t] = order_key(s[i]);
        n_eq += keys[t] == vstar;
      }
    }
    int eq_tot;
    int eq_rank = eq_base + block_exclusive_scan(n_eq, scan_sh, &eq_tot);
    bool keep[SEL_ITEMS];
    int n_keep = 0;
#pragma unroll
    for (int t = 0; t < SEL_ITEMS; ++t) {
      const int i = i_first + t;
      bool kp = false;
      if (i < T) {
        if (keep_all || i < mid_lo || i >= mid_hi) {
          kp = true;
        } else if (k > 0) {
          if (keys[t] > vstar) kp = true;
          else if (keys[t] == vstar) { kp = eq_rank < remaining; ++eq_rank; }
        }
      }
      keep[t] = kp;
      n_keep += kp;
    }
    int keep_tot;
    int pos = base + block_exclusive_scan(n_keep, scan_sh, &keep_tot);
#pragma unroll
    for (int t = 0; t < SEL_ITEMS; ++t)
      if (keep[t]) {
        if (pos < b_max) out[pos] = i_first + t;
        ++pos;
      }
    base += keep_tot;
    eq_base += eq_tot;
  }
  for (int m = base + threadIdx.x; m < b_max; m += blockDim.x) out[m] = -1;
  if (threadIdx.x == 0) {
    count[r] = base;
    if (base != b_eff) raise_status(status, KVP_ERR_DEVICE_CHECK);
  }
}

// ---------------------------------------------------------------------------
constexpr int ST_THREADS = 1024;

__device__ __forceinline__ double st_threshold(double S1, double S2, double k, int m) {
  const double a = k - (double)m;
  if (a >= 0.0) return log(S2 / (sqrt(a * a + S1 * S2) + a));
  return log((sqrt(a * a + S1 * S2) - a) / S1);
}

__global__ void __launch_bounds__(ST_THREADS) soft_topk_kernel(const double* __restrict__ x, int n,
                                                               double k, int t,
                                                               double* __restrict__ ratios,
                                                               int32_t* __restrict__ budgets) {
  __shared__ double xs[ST_THREADS];
  __shared__ double S1[ST_THREADS + 1], S2[ST_THREADS + 1];
  __shared__ double best_v[32];
  __shared__ int best_m[32];
  __shared__ double lam_sh;
  const int tid = threadIdx.x;
  xs[tid] = tid < n ? x[tid] : -INFINITY;
  __syncthreads();
  // Bitonic sort, descending.
  for (int size = 2; size <= ST_THREADS; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int p = tid ^ stride;
      if (p > tid) {
        const bool desc = (tid & size) == 0;
        const double a = xs[tid], c = xs[p];
        if (desc ? (a < c) : (a > c)) { xs[tid] = c; xs[p] = a; }
      }
      __syncthreads();
    }
  }
  if (tid == 0) {
    S1[0] = 0.0;
    for (int m = 0; m < n; ++m) S1[m + 1] = S1[m] + exp(-xs[m]);
    S2[n] = 0.0;
    for (int m = n - 1; m >= 0; --m) S2[m] = S2[m + 1] + exp(xs[m]);
  }
  __syncthreads();
  // Every split m in [0, n]: violation of "top m scores at or above lambda_m, the rest below".
  double v = INFINITY, lam = 0.0;
  int mm = 0x7fffffff;
  for (int m = tid; m <= n; m += blockDim.x) {
    const double l = st_threshold(S1[m], S2[m], k, m);
    const double upper = m > 0 ? xs[m - 1] : INFINITY;
    const double lower = m < n ? xs[m] : -INFINITY;
    const double viol = fmax(0.0, l - upper) + fmax(0.0, lower - l);
    if (viol < v) { v = viol; mm = m; lam = l; }
  }
  // Block argmin over (violation, m).
  for (int o = 16; o > 0; o >>= 1) {
    const double ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int om = __shfl_xor_sync(0xffffffffu, mm, o);
    const double ol = __shfl_xor_sync(0xffffffffu, lam, o);
    if (ov < v || (ov == v && om < mm)) { v = ov; mm = om; lam = ol; }
  }
  if ((tid & 31) == 0) { best_v[tid >> 5] = v; best_m[tid >> 5] = mm; }
  __syncthreads();
  if (tid == 0) {
    int bw = 0;
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
      if (best_v[w] < best_v[bw] || (best_v[w] == best_v[bw] && best_m[w] < best_m[bw])) bw = w;
    const int m = best_m[bw];
    lam_sh = st_threshold(S1[m], S2[m], k, m);
  }
  __syncthreads();
  if (tid < n) {
    const double d = x[tid] - lam_sh;
    const double r = d >= 0.0 ? 1.0 - 0.5 * exp(-d) : 0.5 * exp(d);
    ratios[tid] = r;
    budgets[tid] = (int32_t)floor(r * (double)t);
  }
}

}  // namespace

cudaError_t launch_select(const float* scores, int R, int T, int64_t row_stride,
                          const int32_t* budgets, int n_sink, int n_recent, int32_t* idx,
                          int b_max, int32_t* count, int* status, cudaStream_t st) {
  count_launches(1);
  select_kernel<<<R, SEL_THREADS, 0, st>>>(scores, T, (long long)row_stride, budgets, n_sink,
                                           n_recent, idx, b_max, count, status);
  return cudaGetLastError();
}

cudaError_t launch_soft_topk(const double* x, int n, double k, int t, double* ratios,
                             int32_t* budgets, cudaStream_t st) {
  count_launches(1);
  soft_topk_kernel<<<1, ST_THREADS, 0, st>>>(x, n, k, t, ratios, budgets);
  return cudaGetLastError();
}

}  // namespace kvp
