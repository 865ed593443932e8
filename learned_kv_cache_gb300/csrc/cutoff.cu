// Running top-k cutoffs of KVpop's sparse attention.
//
// KVpop -- Key-Value Cache Compression with Predictive Online Pruning, "Efficient Online
// Pruning" and "Fenwick-tree cut-off computation (Algorithm 2)": at query q the token
// t = q - w leaves the protected window and, unless it is one of the first s sinks, becomes
// eligible; once k tokens are eligible, tau_q is the k-th smallest static rank among them
// (tau_q = -1 before).  The page keeps the eligible ranks in a Fenwick tree and walks the
// queries in order.  Here the same cutoffs come from a bitmap over the ranks, and the query
// axis is cut into chunks that run in parallel:
//
//  * a CTA (head, chunk [q0, q0 + 8 * SUB)) sets the bits of every rank already eligible
//    before q0 (the static set A) and the per-word prefix counts of that bitmap;
//  * each of its 8 warps walks SUB of the chunk's queries in order.  The set at query q is A
//    plus the chunk's ranks inserted up to q (a short list with insertion order), so warps
//    do not interfere.  A warp's first cutoff is found by a binary search on the rank axis
//    (bitmap prefix count + a count over the list); then inserting a rank above the cutoff
//    changes nothing, inserting one below it moves the cutoff to the largest member below
//    the old cutoff (previous set bit of A, or the largest earlier list entry below it), and
//    when the k-th token arrives the cutoff is the largest member.
//
// Repeated or out-of-range ranks are detected and reported through the device status.
#include <climits>

#include "kvp_common.cuh"
#include "kvp_launch.h"

namespace kvp {
namespace {

constexpr int CT_WARPS = 8;
constexpr int CT_THREADS = 32 * CT_WARPS;
// Queries walked by one warp (SUB) is a trade: shorter walks finish sooner, but every CTA
// rebuilds the bitmap of the ranks eligible before its chunk (work ~ S per CTA).  Measured on
// 8 heads: S = 8192 takes 52 / 29 / 21 us with SUB = 64 / 32 / 16, S = 131072 279 / 359 / 607 us.
__host__ __device__ constexpr int ct_chunk(int sub) { return CT_WARPS * sub; }

// Largest set bit of the bitmap < limit, or -1 (warp-uniform).
__device__ __forceinline__ int warp_prev_bit(const uint32_t* bits, int limit, int lane) {
  if (limit <= 0) return -1;
  const int w0 = (limit - 1) >> 5;
  const int nb = limit - (w0 << 5);                    // bits of word w0 below the limit (1..32)
  const uint32_t first = bits[w0] & (nb == 32 ? 0xffffffffu : ((1u << nb) - 1u));
  if (first) return (w0 << 5) + 31 - __clz(first);
  for (int base = w0 - 1; base >= 0; base -= 32) {
    const int wi = base - lane;
    const uint32_t v = wi >= 0 ? bits[wi] : 0u;
    const uint32_t bal = __ballot_sync(0xffffffffu, v != 0u);
    if (bal) {
      const int src = __ffs(bal) - 1;                  // nearest word below
      const uint32_t word = __shfl_sync(0xffffffffu, v, src);
      return ((base - src) << 5) + 31 - __clz(word);
    }
  }
  return -1;
}

// Largest list entry ins[j] < limit with j < n (entries < 0 are not ranks), or -1.
__device__ __forceinline__ int warp_prev_listed(const int* ins, int n, int limit) {
  int best = -1;
  for (int j = threadIdx.x & 31; j < n; j += 32) {
    const int r = ins[j];
    if (r < limit && r > best) best = r;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
  return best;
}

// Number of list entries 0 <= ins[j] <= x with j < n.
__device__ __forceinline__ int warp_count_listed(const int* ins, int n, int x) {
  int c = 0;
  for (int j = threadIdx.x & 31; j < n; j += 32) {
    const int r = ins[j];
    c += (r >= 0 && r <= x) ? 1 : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  return c;
}

template <int CT_SUB>
__global__ void __launch_bounds__(CT_THREADS) cutoff_kernel(const int32_t* __restrict__ ranks, int S,
                                                           int n_sink, int window, int k,
                                                           int32_t* __restrict__ tau, int* status) {
  constexpr int CT_CHUNK = ct_chunk(CT_SUB);        // queries per CTA
  extern __shared__ uint32_t sm[];
  const int nw = (S + 31) >> 5;
  uint32_t* bits = sm;                                       // [nw] the static set A
  int* wpre = reinterpret_cast<int*>(bits + nw);             // [nw] set bits in words before i
  int* cnt = wpre + nw;                                      // [CT_THREADS]
  int* ins = cnt + CT_THREADS;                               // [CT_CHUNK] rank inserted at q0 + i
  int* out = ins + CT_CHUNK;                                 // [CT_CHUNK]
  __shared__ int bad_sh, maxA_sh;
  const int h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q0 = blockIdx.x * CT_CHUNK;
  if (q0 >= S) return;
  const int q1 = min(S, q0 + CT_CHUNK);
  const int32_t* rh = ranks + (size_t)h * S;

  for (int i = tid; i < nw; i += CT_THREADS) bits[i] = 0u;
  if (tid == 0) bad_sh = 0;
  __syncthreads();
  // A: ranks of tokens s .. q0 - 1 - w
  const long long t_last = (long long)q0 - 1 - window;
  int bad = 0;
  for (long long t = n_sink + tid; t <= t_last; t += CT_THREADS) {
    const int r = rh[t];
    if ((unsigned)r < (unsigned)S) {
      const uint32_t bit = 1u << (r & 31);
      if (atomicOr(&bits[r >> 5], bit) & bit) bad = 1;   // repeated rank
    } else {
      bad = 1;
    }
  }
  for (int i = tid; i < CT_CHUNK; i += CT_THREADS) {
    const long long t = (long long)(q0 + i) - window;
    int r = -1;                                              // no insert at this query
    if (q0 + i < q1 && t >= n_sink) {
      r = rh[t];
      if ((unsigned)r >= (unsigned)S) {
        bad = 1;
        r = -1;
      }
    }
    ins[i] = r;
  }
  __syncthreads();                                           // A is complete
  // per-word prefix counts of A
  const int per = (nw + CT_THREADS - 1) / CT_THREADS;
  const int wa = min(nw, tid * per), wb = min(nw, wa + per);
  int c = 0;
  for (int i = wa; i < wb; ++i) c += __popc(bits[i]);
  cnt[tid] = c;
  __syncthreads();
  for (int off = 1; off < CT_THREADS; off <<= 1) {            // inclusive scan (Hillis-Steele)
    const int add = tid >= off ? cnt[tid - off] : 0;
    __syncthreads();
    cnt[tid] += add;
    __syncthreads();
  }
  {
    int run = tid ? cnt[tid - 1] : 0;
    for (int i = wa; i < wb; ++i) {
      wpre[i] = run;
      run += __popc(bits[i]);
    }
  }
  const long long e0 = t_last >= n_sink ? t_last - n_sink + 1 : 0;   // |A| if ranks are valid
  if (tid == CT_THREADS - 1 && (long long)cnt[tid] != e0) bad = 1;
  if (bad) bad_sh = 1;
  __syncthreads();
  if (warp == 0) {
    const int m = warp_prev_bit(bits, S, lane);
    if (lane == 0) maxA_sh = m;
  }
  __syncthreads();

  // walk of this warp's queries [qa, qb)
  const int ia = warp * CT_SUB, ib = min(q1 - q0, ia + CT_SUB);
  if (ia < ib) {
    int before = 0;                                          // inserts of the earlier warps
    for (int j = lane; j < ia; j += 32) before += ins[j] >= 0 ? 1 : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
    long long e = e0 + before;
    int cur = -1;
    if (e >= k) {
      // smallest x with |A <= x| + |list[0, ia) <= x| >= k
      int lo = 0, hi = S - 1;
      while (lo < hi) {
        const int x = (lo + hi) >> 1;
        const int wx = x >> 5, bx = x & 31;
        const uint32_t upto = bx == 31 ? 0xffffffffu : ((2u << bx) - 1u);
        const int cA = wpre[wx] + __popc(bits[wx] & upto);
        if ((long long)cA + warp_count_listed(ins, ia, x) >= k) hi = x;
        else lo = x + 1;
      }
      cur = lo;
    }
    for (int i = ia; i < ib; ++i) {
      const int r = ins[i];
      if (r >= 0) {
        ++e;
        if (e == k) {
          cur = max(maxA_sh, warp_prev_listed(ins, i + 1, INT_MAX));
        } else if (e > k && r < cur) {
          cur = max(warp_prev_bit(bits, cur, lane), warp_prev_listed(ins, i + 1, cur));
        }
      }
      if (lane == 0) out[i] = e >= k ? cur : -1;
    }
  }
  __syncthreads();
  // the chunk's ranks must be new and distinct
  for (int i = tid; i < q1 - q0; i += CT_THREADS) {
    const int r = ins[i];
    if (r >= 0) {
      const uint32_t bit = 1u << (r & 31);
      if (atomicOr(&bits[r >> 5], bit) & bit) bad_sh = 1;
    }
    tau[(size_t)h * S + q0 + i] = out[i];
  }
  __syncthreads();
  if (tid == 0 && bad_sh) raise_status(status, KVP_ERR_DEVICE_CHECK);
}

template <int SUB>
cudaError_t launch_cutoffs_sub(const int32_t* ranks, int n_heads, int S, int n_sink, int window, int k,
                               int32_t* tau, int* status, cudaStream_t st) {
  const int nw = (S + 31) >> 5;
  const size_t smem = (2 * (size_t)nw + CT_THREADS + 2 * ct_chunk(SUB)) * 4;
  cudaError_t e = cudaFuncSetAttribute(cutoff_kernel<SUB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((S + ct_chunk(SUB) - 1) / ct_chunk(SUB), n_heads);
  count_launches(1);
  cutoff_kernel<SUB><<<grid, CT_THREADS, smem, st>>>(ranks, S, n_sink, window, k, tau, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_topk_cutoffs(const int32_t* ranks, int n_heads, int S, int n_sink, int window,
                                int k, int32_t* tau, int* status, cudaStream_t st) {
  if (S <= 16384) return launch_cutoffs_sub<16>(ranks, n_heads, S, n_sink, window, k, tau, status, st);
  if (S <= 65536) return launch_cutoffs_sub<32>(ranks, n_heads, S, n_sink, window, k, tau, status, st);
  return launch_cutoffs_sub<64>(ranks, n_heads, S, n_sink, window, k, tau, status, st);
}

}  // namespace kvp
