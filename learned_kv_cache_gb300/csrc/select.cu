// Budgeted selection (sinks + recent window + top-k) and Soft-TopK head budgets.
//
// Selection (KVpop "The KVpop Scoring Module"; Learning to Evict from
// Key-Value Cache §A.2; How much KV cache can you prune "What we did"):
// scores are mapped to order-preserving uint32 keys (NaN lowest, -0.0 folded
// onto +0.0); a 4-pass 8-bit radix select finds the k-th largest key v* and
// how many of the keys equal to v* must be kept; a final pass in token order
// keeps keys > v*, the first `remaining` keys == v* (lowest indices first) and
// the sinks / recent window, and writes their indices in ascending order
// through block-wide prefix scans.
//
// A row is handled by a thread-block cluster of up to 8 CTAs: each CTA keeps
// the keys of its slice of the row in shared memory (one read of the scores
// from HBM), the per-pass histograms are summed across the cluster through
// distributed shared memory, and the tie ranks and output offsets come from
// cluster-wide prefix counts.  Rows longer than 8 slices of shared memory use
// the single-CTA kernel, which re-reads the row from L2 on every pass.
//
// Soft-TopK (LKV "The Differentiable Soft-TopK Operator", "LKV-H"): one CTA
// sorts the n <= 1024 head scores, forms the prefix sums S1 = sum exp(-x) and
// suffix sums S2 = sum exp(x), evaluates the closed-form threshold for every
// split m and keeps the split that is consistent (top m scores at or above
// the threshold); ratios are the Laplace CDF of (x - lambda), b = floor(r*t).
#include <cooperative_groups.h>
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


// Add 1 to hist[bin] for every active lane, one atomic per distinct bin per warp.
__device__ __forceinline__ void hist_add(int* hist, uint32_t bin, bool active) {
  const unsigned act = __ballot_sync(0xffffffffu, active);
  if (!active) return;
  const unsigned peers = __match_any_sync(act, bin);
  if ((int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
}

// Warp 0: the digit d whose bin holds the `remaining`-th largest key (bins scanned from 255
// down), and how many keys of that bin are still needed.
__device__ __forceinline__ void pick_digit(const int* hist, int remaining, int* sel_digit, int* sel_rem) {
  const int lane = threadIdx.x & 31;
  int c[8], sum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    c[j] = hist[255 - 8 * lane - j];
    sum += c[j];
  }
  const int inc = warp_inclusive_scan(sum);
  const unsigned ball = __ballot_sync(0xffffffffu, inc >= remaining);
  const int L = ball ? __ffs(ball) - 1 : 31;
  if (lane == L) {
    int cum = inc - sum, d = 255 - 8 * lane - 7, rem = remaining - (inc - c[7]);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (cum + c[j] >= remaining) {
        d = 255 - 8 * lane - j;
        rem = remaining - cum;
        break;
      }
      cum += c[j];
    }
    *sel_digit = d;
    *sel_rem = rem;
  }
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
      for (int i0 = mid_lo; i0 < mid_hi; i0 += blockDim.x) {
        const int i = i0 + threadIdx.x;
        const uint32_t key = i < mid_hi ? order_key(s[i]) : 0u;
        hist_add(hist, (key >> shift) & 255u, i < mid_hi && (key & mask) == prefix);
      }
      __syncthreads();
      if (threadIdx.x < 32) pick_digit(hist, remaining, &sel_digit, &sel_remaining);
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
constexpr int SC_THREADS = 512;
constexpr int SC_ITEMS = 4;
constexpr int SC_MAX_SLICE = 16384;       // keys of one CTA's slice held in shared memory
constexpr int SC_MAX_CLUSTER = 8;

__global__ void __launch_bounds__(SC_THREADS) select_cluster_kernel(
    const float* __restrict__ scores, int T, long long row_stride, const int32_t* __restrict__ budgets,
    int n_sink, int n_recent, int32_t* __restrict__ idx, int b_max, int32_t* __restrict__ count,
    int* status) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int r = blockIdx.x / CL;
  extern __shared__ uint32_t keys[];
  __shared__ int hist[2][256];
  __shared__ int hsum[256];
  __shared__ int pub[2];                 // published counts: [0] ties, [1] kept
  __shared__ int scan_sh[33];
  __shared__ int sel_digit, sel_rem;
  const int tid = threadIdx.x;

  const float* s = scores + (size_t)r * row_stride;
  int32_t* out = idx + (size_t)r * b_max;
  const int b = budgets[r];
  const int b_eff = b < 0 ? -1 : ((T <= b) ? T : min(T, max(b, n_sink + n_recent)));
  if (b < 0 || b_eff > b_max) {          // every CTA of the cluster takes this exit
    if (rank == 0 && tid == 0) {
      count[r] = -1;
      raise_status(status, KVP_ERR_DEVICE_CHECK);
    }
    return;
  }
  const bool keep_all = b_eff >= T;
  const int mid_lo = n_sink, mid_hi = T - n_recent;
  const int k = keep_all ? 0 : b_eff - n_sink - n_recent;
  const int per = (T + CL - 1) / CL;
  const int lo = min(T, rank * per), hi = min(T, lo + per);
  const int nloc = hi - lo;
  if (k > 0) {
    // 8 independent loads in flight per thread before the keys are stored
    constexpr int U = 8;
    for (int i0 = 0; i0 < nloc; i0 += U * SC_THREADS) {
      float v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * SC_THREADS + tid;
        v[u] = i < nloc ? __ldg(s + lo + i) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * SC_THREADS + tid;
        if (i < nloc) keys[i] = order_key(v[u]);
      }
    }
  }

  uint32_t prefix = 0u, mask = 0u;
  int remaining = k;
  if (k > 0) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      int* h = hist[pass & 1];
      for (int i = tid; i < 256; i += blockDim.x) h[i] = 0;
      __syncthreads();
      for (int i0 = 0; i0 < nloc; i0 += blockDim.x) {
        const int i = i0 + tid, gi = lo + i;
        const bool in = i < nloc && gi >= mid_lo && gi < mid_hi;
        const uint32_t key = in ? keys[i] : 0u;
        hist_add(h, (key >> shift) & 255u, in && (key & mask) == prefix);
      }
      cluster.sync();
      for (int i = tid; i < 256; i += blockDim.x) {
        int tot = 0;
        for (int qr = 0; qr < CL; ++qr) tot += cluster.map_shared_rank(h, qr)[i];
        hsum[i] = tot;
      }
      __syncthreads();
      if (tid < 32) pick_digit(hsum, remaining, &sel_digit, &sel_rem);
      __syncthreads();
      prefix |= (uint32_t)sel_digit << shift;
      mask |= 255u << shift;
      remaining = sel_rem;
    }
  }
  const uint32_t vstar = prefix;

  // Slice totals: ties (keys == v* in the middle), then kept tokens.
  int n_eq = 0, n_gt = 0, n_fixed = 0;
  for (int i = tid; i < nloc; i += blockDim.x) {
    const int gi = lo + i;
    if (keep_all || gi < mid_lo || gi >= mid_hi) {
      ++n_fixed;
    } else if (k > 0) {
      n_eq += keys[i] == vstar;
      n_gt += keys[i] > vstar;
    }
  }
  int tot;
  block_exclusive_scan(n_eq, scan_sh, &tot);
  n_eq = tot;
  block_exclusive_scan(n_gt, scan_sh, &tot);
  n_gt = tot;
  block_exclusive_scan(n_fixed, scan_sh, &tot);
  n_fixed = tot;
  if (tid == 0) pub[0] = n_eq;
  cluster.sync();
  int eq_before = 0;
  for (int qr = 0; qr < rank; ++qr) eq_before += *cluster.map_shared_rank(&pub[0], qr);
  const int eq_keep = k > 0 ? max(0, min(n_eq, remaining - eq_before)) : 0;
  if (tid == 0) pub[1] = n_fixed + n_gt + eq_keep;
  cluster.sync();
  int base = 0;
  for (int qr = 0; qr < rank; ++qr) base += *cluster.map_shared_rank(&pub[1], qr);
  int total_kept = 0;
  for (int qr = 0; qr < CL; ++qr) total_kept += *cluster.map_shared_rank(&pub[1], qr);
  cluster.sync();                        // no CTA leaves while others read its counts

  // Write the kept indices of this slice in token order.
  int eq_base = eq_before;
  for (int c0 = 0; c0 < nloc; c0 += SC_THREADS * SC_ITEMS) {
    const int i_first = c0 + tid * SC_ITEMS;
    int ne = 0;
#pragma unroll
    for (int t = 0; t < SC_ITEMS; ++t) {
      const int i = i_first + t, gi = lo + i;
      if (k > 0 && i < nloc && gi >= mid_lo && gi < mid_hi) ne += keys[i] == vstar;
    }
    int etot;
    int eq_rank = eq_base + block_exclusive_scan(ne, scan_sh, &etot);
    bool kp[SC_ITEMS];
    int nk = 0;
#pragma unroll
    for (int t = 0; t < SC_ITEMS; ++t) {
      const int i = i_first + t, gi = lo + i;
      bool v = false;
      if (i < nloc) {
        if (keep_all || gi < mid_lo || gi >= mid_hi) {
          v = true;
        } else if (k > 0) {
          if (keys[i] > vstar) v = true;
          else if (keys[i] == vstar) { v = eq_rank < remaining; ++eq_rank; }
        }
      }
      kp[t] = v;
      nk += v;
    }
    int ktot;
    int pos = base + block_exclusive_scan(nk, scan_sh, &ktot);
#pragma unroll
    for (int t = 0; t < SC_ITEMS; ++t)
      if (kp[t]) {
        if (pos < b_max) out[pos] = lo + i_first + t;
        ++pos;
      }
    base += ktot;
    eq_base += etot;
  }
  for (int m = total_kept + rank * blockDim.x + tid; m < b_max; m += CL * blockDim.x) out[m] = -1;
  if (rank == 0 && tid == 0) {
    count[r] = total_kept;
    if (total_kept != b_eff) raise_status(status, KVP_ERR_DEVICE_CHECK);
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
  int cl = 1;
  while (cl < SC_MAX_CLUSTER && T / (2 * cl) >= 1024) cl *= 2;
  const int per = (T + cl - 1) / cl;
  if (per > SC_MAX_SLICE) {
    count_launches(1);
    select_kernel<<<R, SEL_THREADS, 0, st>>>(scores, T, (long long)row_stride, budgets, n_sink,
                                             n_recent, idx, b_max, count, status);
    return cudaGetLastError();
  }
  const size_t smem = (size_t)per * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(select_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(R * cl));
  cfg.blockDim = dim3(SC_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launches(1);
  e = cudaLaunchKernelEx(&cfg, select_cluster_kernel, scores, T, (long long)row_stride, budgets, n_sink,
                         n_recent, idx, b_max, count, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_soft_topk(const double* x, int n, double k, int t, double* ratios,
                             int32_t* budgets, cudaStream_t st) {
  count_launches(1);
  soft_topk_kernel<<<1, ST_THREADS, 0, st>>>(x, n, k, t, ratios, budgets);
  return cudaGetLastError();
}

}  // namespace kvp
