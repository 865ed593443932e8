// Budgeted selection (sinks + recent window + top-k) and Soft-TopK head budgets.
//
// Selection (KVpop "The KVpop Scoring Module"; Learning to Evict from
// Key-Value Cache §A.2; How much KV cache can you prune "What we did"):
// scores are mapped to order-preserving uint32 keys (NaN lowest, -0.0 folded
// onto +0.0); the k-th largest key v* and how many of the keys equal to v*
// must be kept are found by an 11-bit histogram of the key bits below the
// row's common prefix, then exactly among the keys of the boundary bin; a
// final pass in token order keeps keys > v*, the first `remaining` keys == v*
// (lowest indices first) and the sinks / recent window, and writes their
// indices in ascending order with warp ballots.  One thread-block cluster of
// up to 8 CTAs per row; histograms and candidates are combined through
// distributed shared memory (details at select_cluster_kernel).
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


// ---------------------------------------------------------------------------
constexpr int SC_THREADS = 512;
constexpr int SC_WARPS = SC_THREADS / 32;
constexpr int SC_MAX_CLUSTER = 8;
constexpr int SC_BITS = 11;                    // digit width of a histogram level
constexpr int SC_BINS = 1 << SC_BITS;          // 2048
constexpr int SC_BPT = SC_BINS / SC_THREADS;   // 4 consecutive bins per thread in the reductions
constexpr int SC_CAP = 4096;                   // boundary-bin keys a CTA can hold as candidates
static_assert(SC_BPT == 4, "one int4 of bins per thread");

struct SelShared {
  int hist[2][SC_BINS];       // this CTA's histogram per level (double-buffered across levels)
  uint32_t ckey[SC_CAP];      // candidates: keys of the boundary bin in this slice ...
  int32_t cidx[SC_CAP];       // ... and their slice-local positions
  uint32_t mm[2][SC_WARPS];
  uint32_t span[2];           // this CTA's smallest / largest middle key
  int pub[3];                 // this slice's fixed (sink / recent) count, keys > v*, keys == v*
  int scan[33];
  int red[SC_WARPS];
  int wk[SC_WARPS], wt[SC_WARPS], wbase[SC_WARPS], wtie[SC_WARPS];
  int ncand;
  int sel_digit, sel_rem, sel_tot;
  int eq_before, base, total;
};

__device__ __forceinline__ int block_sum(int v, int* red) {
  v = __reduce_add_sync(0xffffffffu, v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  int t = 0;
#pragma unroll
  for (int w = 0; w < SC_WARPS; ++w) t += red[w];
  __syncthreads();
  return t;
}

// The boundary digit of a level: bins are scanned from the top (thread t holds the four bins
// SC_BINS-4t-1 .. SC_BINS-4t-4, totals tot[0..3] in that order); the bin that holds the
// `remaining`-th largest key, how many keys of it are still needed, and its total.
__device__ __forceinline__ void pick_boundary(const int (&tot)[SC_BPT], int remaining, SelShared& sh) {
  const int sum = tot[0] + tot[1] + tot[2] + tot[3];
  int all;
  const int excl = block_exclusive_scan(sum, sh.scan, &all);
  if (excl < remaining && excl + sum >= remaining) {
    int cum = excl;
#pragma unroll
    for (int j = 0; j < SC_BPT; ++j) {
      if (cum + tot[j] >= remaining) {
        sh.sel_digit = SC_BINS - 1 - SC_BPT * (int)threadIdx.x - j;
        sh.sel_rem = remaining - cum;
        sh.sel_tot = tot[j];
        break;
      }
      cum += tot[j];
    }
  }
  __syncthreads();
}

// The scores of a row are entries 0..T-1 of the concatenation of two sources: positions
// gi < n_a come from `scores` (row stride row_stride), the rest from `scores_b` (row stride
// row_stride_b) at gi - n_a.  One source: n_a = T.  budgets == null: every row's budget is
// b_uniform.
//
// One thread-block cluster of up to 8 CTAs per row, each owning a contiguous slice; the scores
// are re-read from L2 on every pass (shared memory holds only histograms and candidates, so
// every cluster of a large launch is resident at once).  With k = b_eff - n_sink - n_recent:
//  1. the smallest and largest middle keys (cluster-wide): the bits they share are common to
//     every middle key, so the levels below start at their highest differing bit;
//  2. levels of an 11-bit histogram of the next digit (summed over the cluster through DSMEM):
//     the digit whose bin holds the k-th largest key is appended to the prefix, the keys in the
//     bins above it are known to be kept; a level stops early once the boundary bin holds at
//     most SC_CAP keys;
//  3. those candidates are gathered per CTA and the exact k-th key v* found among them by
//     further digits (every CTA of the cluster, redundantly, over DSMEM);
//  4. per-slice counts of fixed, > v* and == v* keys give each slice its tie ranks and output
//     offset; two warp-chunked passes in token order (counts, then ballot-ranked writes) emit
//     the kept indices ascending.
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
  extern __shared__ __align__(16) uint8_t sc_raw[];
  SelShared& sh = *reinterpret_cast<SelShared*>(sc_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  wait_prior_grid();                     // the scores may come from the kernel just before

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
  const int mid_lo = n_sink, mid_hi = T - n_recent;     // not keep_all: n_sink + n_recent < T
  const int k = keep_all ? 0 : b_eff - n_sink - n_recent;
  // Slices start at multiples of 4 keys: a slice of a 16-byte aligned single-source row is read
  // with 16-byte loads, four keys per load (otherwise four scalar loads).
  const int per = (((T + CL - 1) / CL) + 3) & ~3;
  const int lo = min(T, rank * per), hi = min(T, lo + per);
  const int nloc = hi - lo;
  const bool vec = scores_b == nullptr && ((reinterpret_cast<uintptr_t>(s + lo) & 15u) == 0);
  // keys of the slice's local positions 4g .. 4g+3 (positions at or past nloc give 0)
  auto keys4 = [&](int g, uint32_t (&kk)[4]) {
    const int i = 4 * g;
    if (vec && i + 3 < nloc) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(s + lo + i));
      kk[0] = order_key(v.x);
      kk[1] = order_key(v.y);
      kk[2] = order_key(v.z);
      kk[3] = order_key(v.w);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) kk[j] = i + j < nloc ? order_key(score_at(lo + i + j)) : 0u;
    }
  };
  // the slice's middle keys are its local positions [mlo, mhi), in the groups [glo, ghi)
  const int mlo = keep_all ? 0 : max(0, min(nloc, mid_lo - lo));
  const int mhi = keep_all ? 0 : max(0, min(nloc, mid_hi - lo));
  const int glo = mlo >> 2, ghi = (mhi + 3) >> 2;

  uint32_t vstar = 0u;
  int rem = 0, gt_local = 0, eq_local = 0;
  if (k > 0) {
    // 1. extremes of the middle keys (the first pass brings the row into L2)
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    {
      constexpr int U = 2;
      for (int g0 = glo; g0 < ghi; g0 += U * SC_THREADS) {
        uint32_t kk[U][4];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int g = g0 + u * SC_THREADS + tid;
          if (g < ghi) keys4(g, kk[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int g = g0 + u * SC_THREADS + tid;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int i = 4 * g + j;
            if (g < ghi && i >= mlo && i < mhi) {
              kmin = min(kmin, kk[u][j]);
              kmax = max(kmax, kk[u][j]);
            }
          }
        }
      }
    }
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    if (lane == 0) {
      sh.mm[0][warp] = kmin;
      sh.mm[1][warp] = kmax;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < SC_WARPS; ++w) {
        kmin = min(kmin, sh.mm[0][w]);
        kmax = max(kmax, sh.mm[1][w]);
      }
      sh.span[0] = kmin;
      sh.span[1] = kmax;
    }
    cluster.sync();
    uint32_t gmin = 0xffffffffu, gmax = 0u;
#pragma unroll
    for (int qr = 0; qr < SC_MAX_CLUSTER; ++qr) {
      if (qr < CL) {
        const uint32_t* rs = cluster.map_shared_rank(&sh.span[0], qr);
        gmin = min(gmin, rs[0]);
        gmax = max(gmax, rs[1]);
      }
    }
    const uint32_t diff = gmin ^ gmax;
    if (diff == 0u) {                      // every middle key is equal: all are ties
      vstar = gmin;
      rem = k;
      eq_local = mhi - mlo;
    } else {
      // 2. histogram levels
      int hib = 31 - __clz(diff);
      uint32_t mask = hib == 31 ? 0u : ~((2u << hib) - 1u);
      uint32_t prefix = gmin & mask;
      int remaining = k;
      bool cand = false;
      for (int lev = 0;; ++lev) {
        const int lob = hib >= SC_BITS - 1 ? hib - (SC_BITS - 1) : 0;
        const uint32_t dmask = (1u << (hib - lob + 1)) - 1u;
        int* h = sh.hist[lev & 1];
        for (int i = tid; i < SC_BINS; i += SC_THREADS) h[i] = 0;
        __syncthreads();
        {
          constexpr int U = 2;
          for (int g0 = glo; g0 < ghi; g0 += U * SC_THREADS) {
            uint32_t kk[U][4];
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const int g = g0 + u * SC_THREADS + tid;
              if (g < ghi) keys4(g, kk[u]);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const int g = g0 + u * SC_THREADS + tid;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int i = 4 * g + j;
                if (g < ghi && i >= mlo && i < mhi && (kk[u][j] & mask) == prefix)
                  atomicAdd(&h[(kk[u][j] >> lob) & dmask], 1);
              }
            }
          }
        }
        cluster.sync();
        int tot[SC_BPT];
        {
          const int bb = SC_BINS - SC_BPT * (tid + 1);
          int4 acc = make_int4(0, 0, 0, 0);
#pragma unroll
          for (int qr = 0; qr < SC_MAX_CLUSTER; ++qr) {
            if (qr < CL) {
              const int4 v = *reinterpret_cast<const int4*>(cluster.map_shared_rank(h, qr) + bb);
              acc.x += v.x;
              acc.y += v.y;
              acc.z += v.z;
              acc.w += v.w;
            }
          }
          tot[0] = acc.w;
          tot[1] = acc.z;
          tot[2] = acc.y;
          tot[3] = acc.x;
        }
        pick_boundary(tot, remaining, sh);
        const int d = sh.sel_digit;
        int above = 0;
        for (int i = tid; i < SC_BINS; i += SC_THREADS) above += i > d ? h[i] : 0;
        gt_local += block_sum(above, sh.red);
        const int at_d = h[d];
        const int bin_tot = sh.sel_tot;
        remaining = sh.sel_rem;
        prefix |= (uint32_t)d << lob;
        mask |= dmask << lob;
        if (lob == 0) {                    // every key of the bin equals v*
          vstar = prefix;
          rem = remaining;
          eq_local = at_d;
          break;
        }
        hib = lob - 1;
        if (bin_tot <= SC_CAP) {
          cand = true;
          break;
        }
      }
      if (cand) {
        // 3. the boundary bin's keys of this slice (at most its cluster total <= SC_CAP)
        if (tid == 0) sh.ncand = 0;
        __syncthreads();
        for (int g = glo + tid; g < ghi; g += SC_THREADS) {
          uint32_t kk[4];
          keys4(g, kk);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int i = 4 * g + j;
            if (i >= mlo && i < mhi && (kk[j] & mask) == prefix) {
              const int slot = atomicAdd(&sh.ncand, 1);
              sh.ckey[slot] = kk[j];
              sh.cidx[slot] = i;
            }
          }
        }
        cluster.sync();
        int nq[SC_MAX_CLUSTER];
#pragma unroll
        for (int qr = 0; qr < SC_MAX_CLUSTER; ++qr) nq[qr] = qr < CL ? *cluster.map_shared_rank(&sh.ncand, qr) : 0;
        // exact digits over the row's candidates (local histograms: no CTA reads them remotely)
        for (int lev = 0;; ++lev) {
          const int lob = hib >= SC_BITS - 1 ? hib - (SC_BITS - 1) : 0;
          const uint32_t dmask = (1u << (hib - lob + 1)) - 1u;
          int* h = sh.hist[lev & 1];
          for (int i = tid; i < SC_BINS; i += SC_THREADS) h[i] = 0;
          __syncthreads();
#pragma unroll
          for (int qr = 0; qr < SC_MAX_CLUSTER; ++qr) {
            if (qr < CL) {
              const uint32_t* ck = cluster.map_shared_rank(sh.ckey, qr);
              for (int i = tid; i < nq[qr]; i += SC_THREADS) {
                const uint32_t key = ck[i];
                if ((key & mask) == prefix) atomicAdd(&h[(key >> lob) & dmask], 1);
              }
            }
          }
          __syncthreads();
          int tot[SC_BPT];
          {
            const int4 v = *reinterpret_cast<const int4*>(h + SC_BINS - SC_BPT * (tid + 1));
            tot[0] = v.w;
            tot[1] = v.z;
            tot[2] = v.y;
            tot[3] = v.x;
          }
          pick_boundary(tot, remaining, sh);
          remaining = sh.sel_rem;
          prefix |= (uint32_t)sh.sel_digit << lob;
          mask |= dmask << lob;
          __syncthreads();
          if (lob == 0) break;
          hib = lob - 1;
        }
        vstar = prefix;
        rem = remaining;
        int g = 0, e = 0;
        for (int i = tid; i < sh.ncand; i += SC_THREADS) {
          const uint32_t key = sh.ckey[i];
          g += key > vstar;
          e += key == vstar;
        }
        gt_local += block_sum(g, sh.red);
        eq_local = block_sum(e, sh.red);
      }
    }
  }

  // 4. slice counts -> tie ranks and output offsets
  const int n_fixed = keep_all ? nloc : nloc - (mhi - mlo);
  if (tid == 0) {
    sh.pub[0] = n_fixed;
    sh.pub[1] = gt_local;
    sh.pub[2] = eq_local;
  }
  cluster.sync();
  if (tid == 0) {
    int eqb = 0, base = 0, total = 0, my_eqb = 0;
    for (int qr = 0; qr < CL; ++qr) {
      const int* pq = cluster.map_shared_rank(&sh.pub[0], qr);
      const int f = pq[0], g = pq[1], e = pq[2];
      const int keep_e = max(0, min(e, rem - eqb));
      if (qr == rank) {
        base = total;
        my_eqb = eqb;
      }
      total += f + g + keep_e;
      eqb += e;
    }
    sh.eq_before = my_eqb;
    sh.base = base;
    sh.total = total;
  }
  __syncthreads();
  const int eq_before = sh.eq_before, total_kept = sh.total;
  // a key's class: 2 kept (sink / recent, or > v*), 1 tie (== v*), 0 dropped (or past the slice)
  const bool sel = k > 0;
  auto klass = [&](int i, uint32_t key) -> int {
    if (i >= nloc) return 0;
    if (i < mlo || i >= mhi) return 2;
    if (!sel) return 0;
    return key > vstar ? 2 : (key == vstar ? 1 : 0);
  };
  // warp w owns the contiguous groups [g0, g1) (a multiple of 32 groups), lane l group g0+32t+l
  const int ng = (nloc + 3) >> 2;
  const int cwg = (((ng + SC_WARPS - 1) / SC_WARPS) + 31) & ~31;
  const int g0 = min(ng, warp * cwg), g1 = min(ng, g0 + cwg);
  auto load_for_output = [&](int g, uint32_t (&kk)[4]) {
    if (g < g1 && sel && 4 * g + 3 >= mlo && 4 * g < mhi) {
      keys4(g, kk);
    } else {
      kk[0] = kk[1] = kk[2] = kk[3] = 0u;
    }
  };
  {
    int nk = 0, nt = 0;
    for (int gb = g0; gb < g1; gb += 32) {
      const int g = gb + lane;
      uint32_t kk[4];
      load_for_output(g, kk);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = g < g1 ? klass(4 * g + j, kk[j]) : 0;
        nk += c == 2;
        nt += c == 1;
      }
    }
    nk = __reduce_add_sync(0xffffffffu, nk);
    nt = __reduce_add_sync(0xffffffffu, nt);
    if (lane == 0) {
      sh.wk[warp] = nk;
      sh.wt[warp] = nt;
    }
  }
  __syncthreads();
  if (tid == 0) {
    int tb = eq_before, ob = sh.base;
    for (int w = 0; w < SC_WARPS; ++w) {
      sh.wtie[w] = tb;
      sh.wbase[w] = ob;
      ob += sh.wk[w] + max(0, min(sh.wt[w], rem - tb));
      tb += sh.wt[w];
    }
  }
  __syncthreads();
  {
    // 128 keys per step in token order (lane-major): warp scans of the per-lane tie and kept
    // counts rank the ties and place the kept indices.
    int tie_rank = sh.wtie[warp], pos = sh.wbase[warp];
    for (int gb = g0; gb < g1; gb += 32) {
      const int g = gb + lane;
      uint32_t kk[4];
      load_for_output(g, kk);
      int c[4], nt = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        c[j] = g < g1 ? klass(4 * g + j, kk[j]) : 0;
        nt += c[j] == 1;
      }
      const int t_incl = warp_inclusive_scan(nt);
      int tr = tie_rank + t_incl - nt, nk = 0;
      bool kept[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        kept[j] = c[j] == 2 || (c[j] == 1 && tr < rem);
        tr += c[j] == 1;
        nk += kept[j];
      }
      const int k_incl = warp_inclusive_scan(nk);
      int p = pos + k_incl - nk;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (kept[j]) {
          if (p < b_max) out[p] = lo + 4 * g + j;
          ++p;
        }
      }
      tie_rank += __shfl_sync(0xffffffffu, t_incl, 31);
      pos += __shfl_sync(0xffffffffu, k_incl, 31);
    }
  }
  for (int m = total_kept + rank * SC_THREADS + tid; m < b_max; m += CL * SC_THREADS) out[m] = -1;
  if (rank == 0 && tid == 0) {
    count[r] = total_kept;
    if (total_kept != b_eff) raise_status(status, KVP_ERR_DEVICE_CHECK);
  }
  cluster.sync();                        // no CTA leaves while others read its shared memory
}

// ---------------------------------------------------------------------------
// Rows of at most 8 x SS_SLICE keys: the upper 16 bits of every order key of a CTA's slice stay
// in shared memory after the one pass that reads the scores, so the radix levels and the output
// pass run on shared memory; only the keys whose upper 16 bits equal the boundary's are read
// again (once, from L2) for the lower 16 bits.
constexpr int SS_THREADS = 512;
constexpr int SS_CTAS_PER_SM = 4;              // (launch bounds; its shared memory allows 4 per SM)
constexpr int SS_WARPS = SS_THREADS / 32;
constexpr int SS_SLICE = 16384;                // keys per CTA (32 KB of 16-bit prefixes)
constexpr int SS_LIST = 2048;                  // boundary-bin keys a row can carry as a list

struct SmemSel {
  uint16_t top[SS_SLICE];     // upper 16 bits of the order key of every key of the slice
  uint32_t lkey[SS_LIST];     // this slice's keys of the upper-16 boundary bin, then the row's
  int32_t lpos[SS_LIST];      // slice positions of this slice's listed keys
  uint32_t gt_bits[SS_SLICE / 32];   // listed keys > v* (bit per slice position)
  uint32_t eq_bits[SS_SLICE / 32];   // listed keys == v*
  int hist[2][256];           // this CTA's 8-bit digit histogram (double-buffered across levels)
  int scan[33];
  int wgt[SS_WARPS], weq[SS_WARPS], wbase[SS_WARPS], wtie[SS_WARPS];
  int pub[3];                 // this slice's fixed (sink / recent) count, keys > v*, keys == v*
  int nlist;
  int sel_digit, sel_rem, sel_tot;
  int total;
};

// h[bin] += 1 for the lanes that hold a bin (bin < 0: none).  The digits start below the bits
// the row's keys share, so the bins of a warp's keys are spread (warp-aggregated increments
// through __match_any_sync measured slower).
__device__ __forceinline__ void ss_count(int* h, int bin) {
  if (bin >= 0) atomicAdd(&h[bin], 1);
}

// Digit of one 8-bit level from the per-bin counts v (thread t < 256 holds bin 255 - t, so the
// scan runs from the top): the bin holding the `remaining`-th largest key, how many of it are
// still needed, and its total.  Returns the digit; `remaining` is updated.
__device__ __forceinline__ int ss_pick(int v, SmemSel& sh, int& remaining, int& bin_total) {
  int all;
  const int excl = block_exclusive_scan(v, sh.scan, &all);
  if (excl < remaining && excl + v >= remaining) {
    sh.sel_digit = 255 - (int)threadIdx.x;
    sh.sel_rem = remaining - excl;
    sh.sel_tot = v;
  }
  __syncthreads();
  const int d = sh.sel_digit;
  remaining = sh.sel_rem;
  bin_total = sh.sel_tot;
  __syncthreads();
  return d;
}

// Cluster-summed level over the CTAs' histograms h.
template <typename Cluster>
__device__ __forceinline__ int ss_level(Cluster& cluster, int CL, SmemSel& sh, const int* h, int& remaining,
                                        int& bin_total) {
  const int tid = threadIdx.x;
  int v = 0;
  if (tid < 256) {
    int part[SC_MAX_CLUSTER];
#pragma unroll
    for (int qr = 0; qr < SC_MAX_CLUSTER; ++qr) part[qr] = qr < CL ? cluster.map_shared_rank(h, qr)[255 - tid] : 0;
#pragma unroll
    for (int qr = 0; qr < SC_MAX_CLUSTER; ++qr) v += part[qr];
  }
  return ss_pick(v, sh, remaining, bin_total);
}

__global__ void __launch_bounds__(SS_THREADS, SS_CTAS_PER_SM) select_smem_kernel(
    const float* __restrict__ scores, int T, long long row_stride, const float* __restrict__ scores_b,
    long long row_stride_b, int n_a, const int32_t* __restrict__ budgets, int b_uniform,
    int n_sink, int n_recent, int32_t* __restrict__ idx, int b_max, int32_t* __restrict__ count,
    int* status) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int r = blockIdx.x / CL;
  extern __shared__ __align__(16) uint8_t ss_raw[];
  SmemSel& sh = *reinterpret_cast<SmemSel*>(ss_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  wait_prior_grid();                     // the scores may come from the kernel just before

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
  const int mid_lo = n_sink, mid_hi = T - n_recent;     // not keep_all: n_sink + n_recent < T
  const int k = keep_all ? 0 : b_eff - n_sink - n_recent;
  const int per = (((T + CL - 1) / CL) + 3) & ~3;       // <= SS_SLICE (checked by the launcher)
  const int lo = min(T, rank * per), hi = min(T, lo + per);
  const int nloc = hi - lo;
  const bool vec = scores_b == nullptr && ((reinterpret_cast<uintptr_t>(s + lo) & 15u) == 0);
  const int mlo = keep_all ? 0 : max(0, min(nloc, mid_lo - lo));
  const int mhi = keep_all ? 0 : max(0, min(nloc, mid_hi - lo));
  auto key_at = [&](int i) { return order_key(score_at(lo + i)); };
  // warp w owns the contiguous positions [c0, c1) (cw a multiple of 128: 4 keys per lane)
  const int cw = (((nloc + SS_WARPS - 1) / SS_WARPS) + 127) & ~127;
  const int c0 = min(nloc, warp * cw), c1 = min(nloc, c0 + cw);

  uint32_t b16 = 0u, vstar = 0u;       // upper 16 bits of v*, and v*
  int rem = 0;
  bool listed = false;
  if (tid < SS_WARPS) {
    sh.wgt[tid] = 0;
    sh.weq[tid] = 0;
  }
  if (k > 0) {
    // A. the slice's keys: upper 16 bits kept in shared memory; digit histogram of bits 31..24
    // of the middle keys
    for (int i = tid; i < 256; i += SS_THREADS) sh.hist[0][i] = 0;
    __syncthreads();
    {
      const int ng = (nloc + 3) >> 2;
      constexpr int U = 4;
      for (int g0 = 0; g0 < ng; g0 += U * SS_THREADS) {
        uint32_t kk[U][4];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int g = g0 + u * SS_THREADS + tid, i = 4 * g;
          if (g < ng) {
            if (vec && i + 3 < nloc) {
              const float4 v = __ldg(reinterpret_cast<const float4*>(s + lo + i));
              kk[u][0] = order_key(v.x);
              kk[u][1] = order_key(v.y);
              kk[u][2] = order_key(v.z);
              kk[u][3] = order_key(v.w);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j) kk[u][j] = i + j < nloc ? key_at(i + j) : 0u;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int g = g0 + u * SS_THREADS + tid;
          if (g < ng) {
            const int i = 4 * g;
            // four prefixes in one 8-byte store (i is a multiple of 4; SS_SLICE too)
            *reinterpret_cast<uint2*>(&sh.top[i]) =
                make_uint2((kk[u][0] >> 16) | (kk[u][1] & 0xffff0000u), (kk[u][2] >> 16) | (kk[u][3] & 0xffff0000u));
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (i + j >= mlo && i + j < mhi) atomicAdd(&sh.hist[0][kk[u][j] >> 24], 1);
          }
        }
      }
    }
    int remaining = k, tot = 0;
    cluster.sync();
    const int dA = ss_level(cluster, CL, sh, sh.hist[0], remaining, tot);
    // B. digit histogram of bits 23..16 over the kept prefixes of the middle keys of bin dA
    for (int i = tid; i < 256; i += SS_THREADS) sh.hist[1][i] = 0;
    __syncthreads();
    {
      constexpr int U = 4;
      for (int i0 = mlo; i0 < mhi; i0 += U * SS_THREADS) {
        uint32_t t[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = i0 + u * SS_THREADS + tid;
          t[u] = i < mhi ? sh.top[i] : 0xffffffffu;
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
          if ((int)(t[u] >> 8) == dA) atomicAdd(&sh.hist[1][t[u] & 0xffu], 1);
      }
    }
    cluster.sync();
    const int dB = ss_level(cluster, CL, sh, sh.hist[1], remaining, tot);
    b16 = ((uint32_t)dA << 8) | (uint32_t)dB;
    // C. per warp chunk: middle keys whose prefix is above b16; the keys of the b16 bin listed
    // with their full keys (read again from L2) when the row's bin fits the list
    listed = tot <= SS_LIST;
    if (tid == 0) sh.nlist = 0;
    __syncthreads();
    {
      int gt = 0;
      for (int i0 = c0; i0 < c1; i0 += 128) {
        const int i = i0 + 4 * lane;
        uint2 t2 = make_uint2(0u, 0u);
        if (i < c1) t2 = *reinterpret_cast<const uint2*>(&sh.top[i]);
        const uint32_t t[4] = {t2.x & 0xffffu, t2.x >> 16, t2.y & 0xffffu, t2.y >> 16};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int ij = i + j;
          if (ij < c1 && ij >= mlo && ij < mhi) {
            gt += t[j] > b16;
            if (listed && t[j] == b16) {
              const int slot = atomicAdd(&sh.nlist, 1);
              sh.lpos[slot] = ij;
            }
          }
        }
      }
      gt = __reduce_add_sync(0xffffffffu, gt);
      if (lane == 0) sh.wgt[warp] = gt;
    }
    __syncthreads();
    const int nl = listed ? sh.nlist : 0;
    for (int e = tid; e < nl; e += SS_THREADS) sh.lkey[e] = key_at(sh.lpos[e]);
    for (int e = tid; e < SS_SLICE / 32; e += SS_THREADS) {
      sh.gt_bits[e] = 0u;
      sh.eq_bits[e] = 0u;
    }
    cluster.sync();
    uint32_t pre = b16 << 16;
    if (listed) {
      // D. the lower 16 bits over the row's listed keys: gathered into registers (at most
      // SS_LIST / SS_THREADS per thread: the row's list holds <= SS_LIST keys), then two local
      // 8-bit levels
      int nq[SC_MAX_CLUSTER], nrow = 0;
#pragma unroll
      for (int qr = 0; qr < SC_MAX_CLUSTER; ++qr) {
        nq[qr] = qr < CL ? *cluster.map_shared_rank(&sh.nlist, qr) : 0;
        nrow += nq[qr];
      }
      uint32_t rk[SS_LIST / SS_THREADS];
#pragma unroll
      for (int u = 0; u < SS_LIST / SS_THREADS; ++u) {
        int e = tid + u * SS_THREADS, qr = 0;
        rk[u] = 0u;
        if (e < nrow) {
#pragma unroll
          for (int q = 0; q < SC_MAX_CLUSTER - 1; ++q)
            if (qr == q && e >= nq[q]) {
              e -= nq[q];
              ++qr;
            }
          rk[u] = cluster.map_shared_rank(sh.lkey, qr)[e];
        }
      }
      for (int lev = 0; lev < 2; ++lev) {
        const int shb = lev == 0 ? 8 : 0;
        const uint32_t pmask = lev == 0 ? 0xffff0000u : 0xffffff00u;
        int* h = sh.hist[lev];
        for (int i = tid; i < 256; i += SS_THREADS) h[i] = 0;
        __syncthreads();
#pragma unroll
        for (int u = 0; u < SS_LIST / SS_THREADS; ++u) {
          const int e = tid + u * SS_THREADS;
          ss_count(h, e < nrow && (rk[u] & pmask) == pre ? (int)((rk[u] >> shb) & 0xffu) : -1);
        }
        __syncthreads();
        const int d = ss_pick(tid < 256 ? h[255 - tid] : 0, sh, remaining, tot);
        pre |= (uint32_t)d << shb;
      }
      vstar = pre;
      // this slice's listed keys: class bits by position and counts per warp chunk
      for (int e = tid; e < nl; e += SS_THREADS) {
        const uint32_t key = sh.lkey[e];
        const int i = sh.lpos[e];
        if (key > vstar) {
          atomicOr(&sh.gt_bits[i >> 5], 1u << (i & 31));
          atomicAdd(&sh.wgt[i / cw], 1);
        } else if (key == vstar) {
          atomicOr(&sh.eq_bits[i >> 5], 1u << (i & 31));
          atomicAdd(&sh.weq[i / cw], 1);
        }
      }
    } else {
      // D. the row's b16 bin is too large for the lists: cluster histograms of the full keys of
      // the bin, read again from L2 (rows whose scores are nearly all equal)
      for (int lev = 0; lev < 2; ++lev) {
        const int shb = lev == 0 ? 8 : 0;
        const uint32_t pmask = lev == 0 ? 0xffff0000u : 0xffffff00u;
        int* h = sh.hist[lev];
        for (int i = tid; i < 256; i += SS_THREADS) h[i] = 0;
        __syncthreads();
        for (int i0 = mlo & ~31; i0 < mhi; i0 += SS_THREADS) {
          const int i = i0 + tid;
          int bin = -1;
          if (i >= mlo && i < mhi && sh.top[i] == b16) {
            const uint32_t key = key_at(i);
            if ((key & pmask) == pre) bin = (int)((key >> shb) & 0xffu);
          }
          ss_count(h, bin);
        }
        cluster.sync();
        const int d = ss_level(cluster, CL, sh, h, remaining, tot);
        pre |= (uint32_t)d << shb;
      }
      vstar = pre;
      int g = 0, q = 0;
      for (int i = c0 + lane; i < c1; i += 32) {
        if (i >= mlo && i < mhi && sh.top[i] == b16) {
          const uint32_t key = key_at(i);
          g += key > vstar;
          q += key == vstar;
        }
      }
      g = __reduce_add_sync(0xffffffffu, g);
      q = __reduce_add_sync(0xffffffffu, q);
      __syncthreads();              // wgt[] of pass C complete before it is added to
      if (lane == 0) {
        sh.wgt[warp] += g;
        sh.weq[warp] += q;
      }
    }
    rem = remaining;
    __syncthreads();
  }

  // slice counts -> tie ranks and output offsets
  const int n_fixed = keep_all ? nloc : nloc - (mhi - mlo);
  if (tid < 32) {
    const int g = lane < SS_WARPS ? sh.wgt[lane] : 0;
    const int q = lane < SS_WARPS ? sh.weq[lane] : 0;
    const int gs = __reduce_add_sync(0xffffffffu, g), qs = __reduce_add_sync(0xffffffffu, q);
    if (lane == 0) {
      sh.pub[0] = n_fixed;
      sh.pub[1] = gs;
      sh.pub[2] = qs;
    }
  }
  cluster.sync();
  if (tid < 32) {
    int f = 0, g = 0, e = 0;
    if (lane < CL) {
      const int* pq = cluster.map_shared_rank(&sh.pub[0], lane);
      f = pq[0];
      g = pq[1];
      e = pq[2];
    }
    const int e_incl = warp_inclusive_scan(e);
    const int keep_e = max(0, min(e, rem - (e_incl - e)));
    const int kept = f + g + keep_e;
    const int k_incl = warp_inclusive_scan(kept);
    const int my_eqb = __shfl_sync(0xffffffffu, e_incl - e, rank);
    const int my_base = __shfl_sync(0xffffffffu, k_incl - kept, rank);
    const int total = __shfl_sync(0xffffffffu, k_incl, 31);
    // per warp chunk: fixed keys (positions outside [mlo, mhi)), > v*, == v*
    const int w0 = min(nloc, lane * cw), w1 = min(nloc, w0 + cw);
    const int wf = lane < SS_WARPS ? (w1 - w0) - max(0, min(w1, mhi) - max(w0, mlo)) : 0;
    const int wq = lane < SS_WARPS ? sh.weq[lane] : 0;
    const int wk = lane < SS_WARPS ? wf + sh.wgt[lane] : 0;
    const int t_incl = warp_inclusive_scan(wq);
    const int tb = my_eqb + t_incl - wq;
    const int wkept = wk + max(0, min(wq, rem - tb));
    const int w_incl = warp_inclusive_scan(wkept);
    if (lane < SS_WARPS) {
      sh.wtie[lane] = tb;
      sh.wbase[lane] = my_base + w_incl - wkept;
    }
    if (lane == 0) sh.total = total;
  }
  __syncthreads();
  const int total_kept = sh.total;
  // E. output in token order: a key's class is 2 kept (sink / recent, or > v*), 1 tie (== v*),
  // 0 dropped; keys of the b16 bin take their class from the bits set above (or from L2).  Lane l
  // holds keys 4l..4l+3 of a 128-key step; four ballots place the kept ones.
  const bool sel = k > 0;
  {
    int tie_rank = sh.wtie[warp], pos = sh.wbase[warp];
    const unsigned lt = (1u << lane) - 1u;
    for (int i0 = c0; i0 < c1; i0 += 128) {
      const int i = i0 + 4 * lane;
      uint2 t2 = make_uint2(0u, 0u);
      if (sel && i < c1) t2 = *reinterpret_cast<const uint2*>(&sh.top[i]);
      const uint32_t t[4] = {t2.x & 0xffffu, t2.x >> 16, t2.y & 0xffffu, t2.y >> 16};
      int c[4];
      if (sel && i0 >= mlo && i0 + 128 <= mhi && i0 + 128 <= c1) {
        // the whole step lies in the middle
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          c[j] = t[j] > b16 ? 2 : 0;
          if (t[j] == b16) {
            const int ij = i + j;
            if (listed) c[j] = (sh.gt_bits[ij >> 5] >> (ij & 31)) & 1u ? 2 : (int)((sh.eq_bits[ij >> 5] >> (ij & 31)) & 1u);
            else {
              const uint32_t key = key_at(ij);
              c[j] = key > vstar ? 2 : (key == vstar ? 1 : 0);
            }
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int ij = i + j;
          if (ij >= c1) c[j] = 0;
          else if (ij < mlo || ij >= mhi) c[j] = 2;
          else if (!sel) c[j] = 0;
          else if (t[j] != b16) c[j] = t[j] > b16 ? 2 : 0;
          else if (listed) c[j] = (sh.gt_bits[ij >> 5] >> (ij & 31)) & 1u ? 2 : (int)((sh.eq_bits[ij >> 5] >> (ij & 31)) & 1u);
          else {
            const uint32_t key = key_at(ij);
            c[j] = key > vstar ? 2 : (key == vstar ? 1 : 0);
          }
        }
      }
      // ties (rare): ranked in token order by a warp scan, kept while their rank is below rem
      const int nt = (c[0] == 1) + (c[1] == 1) + (c[2] == 1) + (c[3] == 1);
      if (__any_sync(0xffffffffu, nt > 0)) {
        const int t_incl = warp_inclusive_scan(nt);
        int tr = tie_rank + t_incl - nt;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (c[j] == 1) {
            c[j] = tr < rem ? 2 : 0;
            ++tr;
          }
        }
        tie_rank += __shfl_sync(0xffffffffu, t_incl, 31);
      }
      unsigned bal[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) bal[j] = __ballot_sync(0xffffffffu, c[j] == 2);
      int p = pos + __popc(bal[0] & lt) + __popc(bal[1] & lt) + __popc(bal[2] & lt) + __popc(bal[3] & lt);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (c[j] == 2) {
          if (p < b_max) out[p] = lo + i + j;
          ++p;
        }
      }
      pos += __popc(bal[0]) + __popc(bal[1]) + __popc(bal[2]) + __popc(bal[3]);
    }
  }
  for (int m = total_kept + rank * SS_THREADS + tid; m < b_max; m += CL * SS_THREADS) out[m] = -1;
  if (rank == 0 && tid == 0) {
    count[r] = total_kept;
    if (total_kept != b_eff) raise_status(status, KVP_ERR_DEVICE_CHECK);
  }
  cluster.sync();                        // no CTA leaves while others read its shared memory
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
  // CTAs per row: as few as let a slice fit shared memory, then doubled while every CTA still
  // fits in one wave and keeps a slice of at least 1024 keys (2048 when there are more than 32
  // rows).  Measured: 8 x 8192 best at 8 CTAs a row (14.3 us; 4: 14.4-16.3 us), 56 x 12288 at
  // 4 (18.4 us; 8: 20.5 us), 256 x 32768 at 2 (51.2 us; 8: 75.8 us, four waves).
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long wave = (long long)SS_CTAS_PER_SM * sms;
  const int min_keys = R <= 32 ? 1024 : 2048;
  int cl = 1;
  while (cl < SC_MAX_CLUSTER && (T + cl - 1) / cl > SS_SLICE) cl *= 2;
  while (cl < SC_MAX_CLUSTER && (long long)R * 2 * cl <= wave && T / (2 * cl) >= min_keys) cl *= 2;
  const int per = (((T + cl - 1) / cl) + 3) & ~3;
  // slices that fit shared memory as 16-bit prefixes: the shared-memory kernel; longer rows:
  // the kernel that re-reads the scores from L2 on every pass
  const bool in_smem = per <= SS_SLICE;
  const void* kern = in_smem ? (const void*)select_smem_kernel : (const void*)select_cluster_kernel;
  const size_t smem = in_smem ? sizeof(SmemSel) : sizeof(SelShared);
  cudaError_t e0 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e0 != cudaSuccess) return e0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(R * cl));
  cfg.blockDim = dim3(in_smem ? SS_THREADS : SC_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attribute();
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  count_launches(1);
  const long long rs = (long long)row_stride, rsb = (long long)row_stride_b;
  const int na = scores_b ? n_a : T;
  cudaError_t e = in_smem
      ? cudaLaunchKernelEx(&cfg, select_smem_kernel, scores, T, rs, scores_b, rsb, na, budgets, b_uniform, n_sink,
                           n_recent, idx, b_max, count, status)
      : cudaLaunchKernelEx(&cfg, select_cluster_kernel, scores, T, rs, scores_b, rsb, na, budgets, b_uniform,
                           n_sink, n_recent, idx, b_max, count, status);
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
