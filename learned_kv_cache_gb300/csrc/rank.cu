// Per-row ranking of scores and the eviction-cost AUC of a ranking.
//
// Learning to Evict from Key-Value Cache §1, §3 and §3.1.1: a ranking of a head's entries
// serves every budget (the top-b are kept), and its cost over all budgets is the area under
// the curve cost(b) = sum of the importance of the entries ranked b or later; the optimal
// ranking orders entries by importance.  KVpop, "Efficient Online Pruning": the static ranks
// of the running top-k mask come from sorting the tokens by a static priority score.
//
// Ranking (rank 0 = highest score, ties to the lower index, NaN last, -0.0 == +0.0) is a
// stable least-significant-digit radix sort of (order key, index) pairs, segmented by row:
// four 8-bit passes, each a histogram kernel (one CTA per 2048-entry tile), a scan kernel (one
// CTA per row: digit-major, tile-minor offsets) and a scatter kernel that ranks a tile's
// entries stably (8 rounds of 256 in entry order; warp peers by __match_any_sync, counts of
// the earlier warps from shared memory).  A last kernel inverts the sorted order into ranks.
//
// AUC: sum over b = 0..T of cost(b) equals sum_t (rank_t + 1) * F_t (each entry is counted
// once for every budget that evicts it), so the area is one weighted sum per (row, ranking).
#include "kvp_common.cuh"
#include "kvp_launch.h"

namespace kvp {
namespace {

constexpr int RK_THREADS = 256;
constexpr int RK_PER_THREAD = 8;
constexpr int RK_TILE = RK_THREADS * RK_PER_THREAD;   // 2048 entries per CTA
constexpr int RK_WARPS = RK_THREADS / 32;

// Ascending order of the key = descending score; NaN (key ~0) last; -0.0 folded into +0.0.
__device__ __forceinline__ uint32_t desc_key(float x) {
  if (x != x) return 0xffffffffu;
  uint32_t u = __float_as_uint(x);
  if ((u << 1) == 0u) u = 0u;
  const uint32_t asc = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ~asc;
}

__device__ __forceinline__ uint32_t key_at(const float* scores, const uint32_t* keys, bool first,
                                           size_t i) {
  return first ? desc_key(scores[i]) : keys[i];
}

__global__ void __launch_bounds__(RK_THREADS) rank_hist_kernel(const float* __restrict__ scores,
                                                              const uint32_t* __restrict__ keys,
                                                              int first, int T, int NB, int shift,
                                                              int* __restrict__ hist) {
  wait_prior_grid();
  __shared__ int h[256];
  const int b = blockIdx.x, r = blockIdx.y, tid = threadIdx.x;
  h[tid] = 0;
  __syncthreads();
  const size_t base = (size_t)r * T;
  const int e0 = b * RK_TILE;
  for (int j = 0; j < RK_PER_THREAD; ++j) {
    const int e = e0 + j * RK_THREADS + tid;
    if (e < T) atomicAdd(&h[(key_at(scores, keys, first, base + e) >> shift) & 255u], 1);
  }
  __syncthreads();
  hist[((size_t)r * NB + b) * 256 + tid] = h[tid];
}

// hist[r][b][d] (counts) -> global start of (tile b, digit d) in row r's sorted order.
__global__ void __launch_bounds__(256) rank_scan_kernel(int NB, int* __restrict__ hist) {
  wait_prior_grid();
  __shared__ int tot[256];
  const int r = blockIdx.x, d = threadIdx.x;
  int* hr = hist + (size_t)r * NB * 256;
  int run = 0;
  for (int b = 0; b < NB; ++b) {
    const int c = hr[b * 256 + d];
    hr[b * 256 + d] = run;
    run += c;
  }
  tot[d] = run;
  __syncthreads();
  for (int off = 1; off < 256; off <<= 1) {                 // inclusive scan of the digit totals
    const int add = d >= off ? tot[d - off] : 0;
    __syncthreads();
    tot[d] += add;
    __syncthreads();
  }
  const int before = d ? tot[d - 1] : 0;
  for (int b = 0; b < NB; ++b) hr[b * 256 + d] += before;
}

__global__ void __launch_bounds__(RK_THREADS) rank_scatter_kernel(
    const float* __restrict__ scores, const uint32_t* __restrict__ keys_in,
    const int32_t* __restrict__ vals_in, int first, int T, int NB, int shift,
    const int* __restrict__ hist, uint32_t* __restrict__ keys_out, int32_t* __restrict__ vals_out) {
  wait_prior_grid();
  __shared__ int start[256];                 // global position of the tile's next entry per digit
  __shared__ int wcnt[RK_WARPS][256];        // per-round counts of each warp
  const int b = blockIdx.x, r = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t base = (size_t)r * T;
  start[tid] = hist[((size_t)r * NB + b) * 256 + tid];
  const int e0 = b * RK_TILE;
  const uint32_t lt = (1u << lane) - 1u;
  for (int j = 0; j < RK_PER_THREAD; ++j) {
    for (int w = 0; w < RK_WARPS; ++w) wcnt[w][tid] = 0;
    __syncthreads();
    const int e = e0 + j * RK_THREADS + tid;
    const bool live = e < T;
    uint32_t key = 0u;
    int val = 0, d = 256 + lane;             // a digit no live entry has: dead lanes match only themselves
    if (live) {
      key = key_at(scores, keys_in, first, base + e);
      val = first ? e : vals_in[base + e];
      d = (int)((key >> shift) & 255u);
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, d);
    if (live && (peers & lt) == 0u) wcnt[warp][d] = __popc(peers);   // the lowest peer reports
    __syncthreads();
    if (live) {
      int pos = start[d] + __popc(peers & lt);
      for (int w = 0; w < warp; ++w) pos += wcnt[w][d];
      keys_out[base + pos] = key;
      vals_out[base + pos] = val;
    }
    __syncthreads();
    int add = 0;
    for (int w = 0; w < RK_WARPS; ++w) add += wcnt[w][tid];
    start[tid] += add;
    __syncthreads();
  }
}

__global__ void rank_invert_kernel(const int32_t* __restrict__ vals, int R, int T,
                                   int32_t* __restrict__ ranks, int* status) {
  wait_prior_grid();
  const long long total = (long long)R * T;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(i / T), p = (int)(i % T);
    const int v = vals[i];
    if (v < 0 || v >= T) {
      raise_status(status, KVP_ERR_DEVICE_CHECK);
      continue;
    }
    ranks[(size_t)r * T + v] = p;
  }
}

// auc[r, m] = sum_t (ranks[r, m, t] + 1) * F[r, t], in two kernels: partial sums over chunks
// of AUC_CHUNK entries (grid chunk x ranking x row), then a fixed-order sum of the partials.
// Each product (rank + 1) * F is split exactly into two fp32 numbers (product and its FMA
// residual; rank + 1 <= 2^24 is exact in fp32) and the terms are added with a compensated
// (two-sum) fp32 pair, also when the pairs of a warp are combined; fp64 (slow on this part) is
// used only for the CTA's last sum and the partials, so the result carries no product rounding
// and no long-sum drift.
constexpr int AUC_THREADS = 256;
constexpr int AUC_CHUNK = 8192;

__device__ __forceinline__ void two_sum_add(float& hi, float& lo, float x) {
  const float s = hi + x;
  const float bp = s - hi;
  const float err = (hi - (s - bp)) + (x - bp);
  hi = s;
  lo += err;
}

__global__ void __launch_bounds__(AUC_THREADS) auc_partial_kernel(const float* __restrict__ F,
                                                                  const int32_t* __restrict__ ranks,
                                                                  int M, int T, int NC, int vec,
                                                                  double* __restrict__ part) {
  wait_prior_grid();
  __shared__ double red[AUC_THREADS / 32];
  const int c = blockIdx.x, m = blockIdx.y, r = blockIdx.z, tid = threadIdx.x;
  const float* f = F + (size_t)r * T;
  const int32_t* rk = ranks + ((size_t)r * M + m) * T;
  const int t0 = c * AUC_CHUNK, t1 = min(T, t0 + AUC_CHUNK);
  float hi = 0.f, lo = 0.f;
  auto add = [&](int rank, float fv) {
    const float a = (float)(rank + 1);
    const float p = a * fv;
    const float e = fmaf(a, fv, -p);          // a * fv = p + e exactly
    two_sum_add(hi, lo, p);
    lo += e;
  };
  if (vec) {                                   // rows 16-byte aligned: 4 entries per load, two loads
    constexpr int STEP = 4 * AUC_THREADS;      // of each array in flight per thread
    for (int t = t0 + 4 * tid; t < t1; t += 2 * STEP) {
      const bool a_full = t + 3 < t1, b_full = t + STEP + 3 < t1;
      int4 ra = make_int4(0, 0, 0, 0), rb = ra;
      float4 fa = make_float4(0.f, 0.f, 0.f, 0.f), fb = fa;
      if (a_full) {
        ra = __ldg(reinterpret_cast<const int4*>(rk + t));
        fa = __ldg(reinterpret_cast<const float4*>(f + t));
      }
      if (b_full) {
        rb = __ldg(reinterpret_cast<const int4*>(rk + t + STEP));
        fb = __ldg(reinterpret_cast<const float4*>(f + t + STEP));
      }
      if (a_full) {
        add(ra.x, fa.x);
        add(ra.y, fa.y);
        add(ra.z, fa.z);
        add(ra.w, fa.w);
      } else {
        for (int u = t; u < t1; ++u) add(__ldg(rk + u), __ldg(f + u));
      }
      if (b_full) {
        add(rb.x, fb.x);
        add(rb.y, fb.y);
        add(rb.z, fb.z);
        add(rb.w, fb.w);
      } else {
        for (int u = t + STEP; u < t1; ++u) add(__ldg(rk + u), __ldg(f + u));
      }
    }
  } else {
    for (int t = t0 + tid; t < t1; t += AUC_THREADS) add(__ldg(rk + t), __ldg(f + t));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, hi, o);
    const float ol = __shfl_xor_sync(0xffffffffu, lo, o);
    two_sum_add(hi, lo, oh);
    lo += ol;
  }
  if ((tid & 31) == 0) red[tid >> 5] = (double)hi + (double)lo;
  __syncthreads();
  if (tid == 0) {
    double s = 0.0;
    for (int w = 0; w < AUC_THREADS / 32; ++w) s += red[w];
    part[((size_t)r * M + m) * NC + c] = s;
  }
}

__global__ void auc_reduce_kernel(const double* __restrict__ part, int RM, int NC,
                                  double* __restrict__ auc) {
  wait_prior_grid();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= RM) return;
  double s = 0.0;
  for (int c = 0; c < NC; ++c) s += part[(size_t)i * NC + c];
  auc[i] = s;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

size_t rank_rows_workspace_size(int R, int T) {
  const size_t n = (size_t)R * T;
  const int NB = (T + RK_TILE - 1) / RK_TILE;
  return 4 * align256(n * 4) + align256((size_t)R * NB * 256 * 4);
}

cudaError_t launch_rank_rows(const float* scores, int R, int T, int32_t* ranks, void* ws,
                             int* status, cudaStream_t st) {
  const size_t n = (size_t)R * T;
  const int NB = (T + RK_TILE - 1) / RK_TILE;
  char* p = (char*)ws;
  uint32_t* ka = (uint32_t*)p;
  int32_t* va = (int32_t*)(p + align256(n * 4));
  uint32_t* kb = (uint32_t*)(p + 2 * align256(n * 4));
  int32_t* vb = (int32_t*)(p + 3 * align256(n * 4));
  int* hist = (int*)(p + 4 * align256(n * 4));
  const dim3 grid(NB, R);
  const uint32_t* kin = nullptr;
  const int32_t* vin = nullptr;
  uint32_t* kout = ka;
  int32_t* vout = va;
  for (int pass = 0; pass < 4; ++pass) {
    const int first = pass == 0, shift = 8 * pass;
    count_launches(3);
    cudaError_t e = launch_with_pdl(rank_hist_kernel, grid, dim3(RK_THREADS), 0, st, scores, kin, first, T, NB,
                                    shift, hist);
    if (e == cudaSuccess) e = launch_with_pdl(rank_scan_kernel, dim3(R), dim3(256), 0, st, NB, hist);
    if (e == cudaSuccess)
      e = launch_with_pdl(rank_scatter_kernel, grid, dim3(RK_THREADS), 0, st, scores, kin, vin, first, T, NB, shift,
                          hist, kout, vout);
    if (e != cudaSuccess) return e;
    kin = kout;
    vin = vout;
    kout = kout == ka ? kb : ka;
    vout = vout == va ? vb : va;
  }
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = ((long long)n + 255) / 256;
  if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
  count_launches(1);
  return launch_with_pdl(rank_invert_kernel, dim3((unsigned)blocks), dim3(256), 0, st, vin, R, T, ranks, status);
}

size_t eviction_auc_workspace_size(int R, int M, int T) {
  const int NC = (T + AUC_CHUNK - 1) / AUC_CHUNK;
  return align256((size_t)R * M * NC * sizeof(double));
}

cudaError_t launch_eviction_auc(const float* F, const int32_t* ranks, int R, int M, int T,
                                double* auc, void* ws, cudaStream_t st) {
  const int NC = (T + AUC_CHUNK - 1) / AUC_CHUNK;
  const int vec = T % 4 == 0 && ((uintptr_t)F & 15) == 0 && ((uintptr_t)ranks & 15) == 0;
  double* part = (double*)ws;
  count_launches(2);
  cudaError_t e = launch_with_pdl(auc_partial_kernel, dim3(NC, M, R), dim3(AUC_THREADS), 0, st, F, ranks, M, T, NC,
                                  vec, part);
  if (e != cudaSuccess) return e;
  const int RM = R * M;
  return launch_with_pdl(auc_reduce_kernel, dim3((RM + 255) / 256), dim3(256), 0, st, (const double*)part, RM, NC,
                         auc);
}

}  // namespace kvp
