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
// A row is handled by a thread-block cluster of up to 8 CTAs, each owning one
// slice of the row: the radix passes start at the highest bit where the row's
// keys differ (cluster-wide min / max), per-pass histograms (private to pairs
// of warps) are summed across the
// cluster through distributed shared memory, and the tie ranks and output
// offsets come from cluster-wide prefix counts.  The order keys of a slice
// (up to 16384) live in shared memory; longer slices recompute the rest from
// the L2-resident scores on every pass.
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

// ---------------------------------------------------------------------------
constexpr int SC_THREADS = 512;
constexpr int SC_MAX_CLUSTER = 8;
constexpr int SC_PRIV = 8;                // private histograms per CTA
constexpr int SC_SMEM_KEYS = 16384;       // order keys of a slice held in shared memory (64 KB)

// The scores of a row are entries 0..T-1 of the concatenation of two sources: positions
// gi < n_a come from `scores` (row stride row_stride), the rest from `scores_b` (row stride
// row_stride_b) at gi - n_a.  One source: n_a = T.  budgets == null: every row's budget is
// b_uniform.
__global__ void __launch_bounds__(SC_THREADS, 4) select_cluster_kernel(
    const float* __restrict__ scores, int T, long long row_stride, const float* __restrict__ scores_b,
    long long row_stride_b, int n_a, const int32_t* __restrict__ budgets, int b_uniform,
    int n_sink, int n_recent, int32_t* __restrict__ idx, int b_max, int32_t* __restrict__ count,
    int* status) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int r = blockIdx.x / CL;
  extern __shared__ uint32_t skeys[];    // [min(slice, SC_SMEM_KEYS)]
  __shared__ int hist[2][256];
  __shared__ int hsum[256];
  __shared__ int priv[SC_PRIV][256];     // histograms private to pairs of warps
  __shared__ uint32_t mm_sh[2][SC_THREADS / 32];
  __shared__ uint32_t span[2];           // this CTA's smallest / largest middle key
  __shared__ int pub[2];                 // published counts: [0] ties, [1] kept
  __shared__ int scan_sh[33];
  __shared__ int sel_digit, sel_rem;
  const int tid = threadIdx.x;

  const float* s = scores + (size_t)r * row_stride;
  const float* s_b = scores_b ? scores_b + (size_t)r * row_stride_b - n_a : nullptr;
  auto score_at = [&](int gi) { return gi < n_a ? __ldg(s + gi) : __ldg(s_b + gi); };
  int32_t* out = idx + (size_t)r * b_max;
  const int b = budgets ? budgets[r] : b_uniform;
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
  // The order keys of the slice are kept in shared memory (up to SC_SMEM_KEYS; keys past
  // that are recomputed from the scores, which stay in L2 after the first pass).
  const int nsm = min(nloc, SC_SMEM_KEYS);
  if (k > 0) {
    constexpr int U = 8;
    for (int i0 = 0; i0 < nsm; i0 += U * SC_THREADS) {
      float v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * SC_THREADS + tid;
        v[u] = i < nsm ? score_at(lo + i) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * SC_THREADS + tid;
        if (i < nsm) skeys[i] = order_key(v[u]);
      }
    }
    __syncthreads();
  }
  auto key_at = [&](int i) { return i < SC_SMEM_KEYS ? skeys[i] : order_key(score_at(lo + i)); };
  uint32_t prefix = 0u, mask = 0u;
  int remaining = k;
  if (k > 0) {
    // The bits above the highest bit where the row's smallest and largest middle keys differ
    // are common to every key: the radix passes start below them.
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    for (int i = tid; i < nloc; i += blockDim.x) {
      const int gi = lo + i;
      if (gi >= mid_lo && gi < mid_hi) {
        const uint32_t key = key_at(i);
        kmin = min(kmin, key);
        kmax = max(kmax, key);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, off));
      kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, off));
    }
    if ((tid & 31) == 0) {
      mm_sh[0][tid >> 5] = kmin;
      mm_sh[1][tid >> 5] = kmax;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
        kmin = min(kmin, mm_sh[0][w]);
        kmax = max(kmax, mm_sh[1][w]);
      }
      span[0] = kmin;
      span[1] = kmax;
    }
    cluster.sync();
    uint32_t gmin = 0xffffffffu, gmax = 0u;
    {
      uint32_t lo_v[SC_MAX_CLUSTER], hi_v[SC_MAX_CLUSTER];
#pragma unroll
      for (int qr = 0; qr < SC_MAX_CLUSTER; ++qr) {
        const uint32_t* rs = cluster.map_shared_rank(&span[0], qr < CL ? qr : 0);
        lo_v[qr] = rs[0];
        hi_v[qr] = rs[1];
      }
#pragma unroll
      for (int qr = 0; qr < SC_MAX_CLUSTER; ++qr) {
        gmin = min(gmin, lo_v[qr]);
        gmax = max(gmax, hi_v[qr]);
      }
    }
    const uint32_t diff = gmin ^ gmax;
    if (diff == 0u) {
      prefix = gmin;                       // every middle key is equal
      mask = 0xffffffffu;
    } else {
      int hi = 31 - __clz(diff);
      mask = hi == 31 ? 0u : ~((2u << hi) - 1u);
      prefix = gmin & mask;
      for (int pass = 0; hi >= 0; ++pass) {
        const int lo_bit = hi >= 7 ? hi - 7 : 0;
        const uint32_t dmask = (1u << (hi - lo_bit + 1)) - 1u;
        int* h = hist[pass & 1];
        for (int i = tid; i < SC_PRIV * 256; i += blockDim.x) (&priv[0][0])[i] = 0;
        __syncthreads();
        int* mine = priv[(tid >> 5) % SC_PRIV];
        constexpr int U = 4;                 // independent loads in flight per thread
        for (int i0 = 0; i0 < nloc; i0 += U * SC_THREADS) {
          uint32_t kk[U];
          bool in[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int i = i0 + u * SC_THREADS + tid, gi = lo + i;
            in[u] = i < nloc && gi >= mid_lo && gi < mid_hi;
            kk[u] = in[u] ? key_at(i) : 0u;
          }
#pragma unroll
          for (int u = 0; u < U; ++u)
            if (in[u] && (kk[u] & mask) == prefix) atomicAdd(&mine[(kk[u] >> lo_bit) & dmask], 1);
        }
        __syncthreads();
        for (int i = tid; i < 256; i += blockDim.x) {
          int tot = 0;
#pragma unroll
          for (int j = 0; j < SC_PRIV; ++j) tot += priv[j][i];
          h[i] = tot;
        }
        cluster.sync();
        if (tid < 256) {                   // all remote loads in flight at once
          int v[SC_MAX_CLUSTER];
#pragma unroll
          for (int qr = 0; qr < SC_MAX_CLUSTER; ++qr) v[qr] = qr < CL ? cluster.map_shared_rank(h, qr)[tid] : 0;
          int tot = 0;
#pragma unroll
          for (int qr = 0; qr < SC_MAX_CLUSTER; ++qr) tot += v[qr];
          hsum[tid] = tot;
        }
        __syncthreads();
        if (tid < 32) pick_digit(hsum, remaining, &sel_digit, &sel_rem);
        __syncthreads();
        prefix |= (uint32_t)sel_digit << lo_bit;
        mask |= dmask << lo_bit;
        remaining = sel_rem;
        hi = lo_bit - 1;
      }
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
      const uint32_t key = key_at(i);
      n_eq += key == vstar;
      n_gt += key > vstar;
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
#pragma unroll
  for (int qr = 0; qr < SC_MAX_CLUSTER; ++qr) {
    const int v = *cluster.map_shared_rank(&pub[0], qr < CL ? qr : 0);
    eq_before += qr < rank ? v : 0;
  }
  const int eq_keep = k > 0 ? max(0, min(n_eq, remaining - eq_before)) : 0;
  if (tid == 0) pub[1] = n_fixed + n_gt + eq_keep;
  cluster.sync();
  int base = 0, total_kept = 0;
#pragma unroll
  for (int qr = 0; qr < SC_MAX_CLUSTER; ++qr) {
    const int v = *cluster.map_shared_rank(&pub[1], qr < CL ? qr : 0);
    base += qr < rank ? v : 0;
    total_kept += qr < CL ? v : 0;
  }
  cluster.sync();                        // no CTA leaves while others read its counts

  // Write the kept indices of this slice in token order: thread t owns one contiguous run,
  // so two block scans give every thread its tie rank and its output position.
  {
    const int run = (nloc + (int)blockDim.x - 1) / (int)blockDim.x;
    const int a = min(nloc, tid * run), z = min(nloc, a + run);
    int ne = 0;
    if (k > 0)
      for (int i = a; i < z; ++i) {
        const int gi = lo + i;
        if (gi >= mid_lo && gi < mid_hi) ne += key_at(i) == vstar;
      }
    int etot;
    int eq_rank = eq_before + block_exclusive_scan(ne, scan_sh, &etot);
    const int eq_first = eq_rank;
    int nk = 0;
    for (int i = a; i < z; ++i) {
      const int gi = lo + i;
      if (keep_all || gi < mid_lo || gi >= mid_hi) {
        ++nk;
      } else if (k > 0) {
        const uint32_t key = key_at(i);
        if (key > vstar) ++nk;
        else if (key == vstar) { nk += eq_rank < remaining; ++eq_rank; }
      }
    }
    int ktot;
    int pos = base + block_exclusive_scan(nk, scan_sh, &ktot);
    eq_rank = eq_first;
    for (int i = a; i < z; ++i) {
      const int gi = lo + i;
      bool v = false;
      if (keep_all || gi < mid_lo || gi >= mid_hi) {
        v = true;
      } else if (k > 0) {
        const uint32_t key = key_at(i);
        if (key > vstar) v = true;
        else if (key == vstar) { v = eq_rank < remaining; ++eq_rank; }
      }
      if (v) {
        if (pos < b_max) out[pos] = gi;
        ++pos;
      }
    }
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
                          int b_max, int32_t* count, int* status, cudaStream_t st,
                          const float* scores_b, int64_t row_stride_b, int n_a, int b_uniform) {
  int cl = 1;
  while (cl < SC_MAX_CLUSTER && T / (2 * cl) >= 1024) cl *= 2;
  const int per = (T + cl - 1) / cl;
  const size_t smem = (size_t)(per < SC_SMEM_KEYS ? per : SC_SMEM_KEYS) * sizeof(uint32_t);
  cudaError_t e0 = cudaFuncSetAttribute(select_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)smem);
  if (e0 != cudaSuccess) return e0;
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
  cudaError_t e;
  count_launches(1);
  e = cudaLaunchKernelEx(&cfg, select_cluster_kernel, scores, T, (long long)row_stride, scores_b,
                         (long long)row_stride_b, scores_b ? n_a : T, budgets, b_uniform, n_sink,
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
