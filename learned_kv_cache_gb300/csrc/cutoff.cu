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
//  * a CTA (head, chunk [q0, q1)) first sets the bits of every rank already eligible before
//    q0 and finds the k-th smallest set bit with a block-wide count (word popcounts and a
//    prefix sum over them);
//  * one warp then walks the chunk's queries in order.  Inserting a rank above the cutoff
//    changes nothing; inserting one below it moves the cutoff to the next set bit below the
//    old cutoff (a ballot over 32 words at a time); when the k-th token arrives the cutoff is
//    the largest set bit.
//
// The output of the chunk is staged in shared memory and written with coalesced stores.
#include <climits>

#include "kvp_common.cuh"
#include "kvp_launch.h"

namespace kvp {
namespace {

constexpr int CT_THREADS = 256;
constexpr int CT_CHUNK = 512;     // queries per CTA

// Largest set bit < limit (limit <= 32 * nw), or -1.  Warp-uniform result.
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

__global__ void __launch_bounds__(CT_THREADS) cutoff_kernel(const int32_t* __restrict__ ranks, int S,
                                                           int n_sink, int window, int k,
                                                           int32_t* __restrict__ tau, int* status) {
  extern __shared__ uint32_t sm[];
  const int nw = (S + 31) >> 5;
  uint32_t* bits = sm;                                       // [nw]
  int* cnt = reinterpret_cast<int*>(bits + nw);              // [CT_THREADS]
  int* rk = cnt + CT_THREADS;                                // [CT_CHUNK] rank inserted at q (or -1)
  int* out = rk + CT_CHUNK;                                  // [CT_CHUNK]
  __shared__ int tau0_sh, bad_sh;
  const int h = blockIdx.y, tid = threadIdx.x;
  const int q0 = blockIdx.x * CT_CHUNK;
  if (q0 >= S) return;
  const int q1 = min(S, q0 + CT_CHUNK);
  const int32_t* rh = ranks + (size_t)h * S;

  for (int i = tid; i < nw; i += CT_THREADS) bits[i] = 0u;
  if (tid == 0) {
    tau0_sh = -1;
    bad_sh = 0;
  }
  __syncthreads();
  // ranks eligible before q0: tokens s .. q0 - 1 - w
  const long long t_last = (long long)q0 - 1 - window;
  int bad = 0;
  for (long long t = n_sink + tid; t <= t_last; t += CT_THREADS) {
    const int r = rh[t];
    if ((unsigned)r < (unsigned)S) atomicOr(&bits[r >> 5], 1u << (r & 31));
    else bad = 1;
  }
  for (int q = q0 + tid; q < q1; q += CT_THREADS) {
    const long long t = (long long)q - window;
    int r = -1;
    if (t >= n_sink) {
      r = rh[t];
      if ((unsigned)r >= (unsigned)S) {
        bad = 1;
        r = -2;
      }
    }
    rk[q - q0] = r;
  }
  if (bad) bad_sh = 1;
  __syncthreads();
  const long long e0 = t_last >= n_sink ? t_last - n_sink + 1 : 0;   // eligible before q0

  if (e0 > 0) {
    // k-th smallest set bit: per-thread word ranges, popcount, exclusive prefix sum (the total
    // also checks that the eligible ranks were distinct)
    const int per = (nw + CT_THREADS - 1) / CT_THREADS;
    const int wa = tid * per, wb = min(nw, wa + per);
    int c = 0;
    for (int i = wa; i < wb; ++i) c += __popc(bits[i]);
    cnt[tid] = c;
    __syncthreads();
    for (int off = 1; off < CT_THREADS; off <<= 1) {          // inclusive scan (Hillis-Steele)
      const int add = tid >= off ? cnt[tid - off] : 0;
      __syncthreads();
      cnt[tid] += add;
      __syncthreads();
    }
    const int before = tid ? cnt[tid - 1] : 0;
    if (tid == CT_THREADS - 1 && cnt[tid] != e0) bad_sh = 1;
    if (e0 >= k && before < k && cnt[tid] >= k) {
      int need = k - before;
      for (int i = wa; i < wb; ++i) {
        uint32_t v = bits[i];
        const int pc = __popc(v);
        if (need > pc) {
          need -= pc;
          continue;
        }
        for (int j = 1; j < need; ++j) v &= v - 1u;         // drop the need-1 lowest set bits
        tau0_sh = (i << 5) + __ffs(v) - 1;
        break;
      }
    }
    __syncthreads();
  }

  if (tid < 32) {
    const int lane = tid;
    int cur = tau0_sh;
    long long e = e0;
    int err = 0;
    for (int q = q0; q < q1; ++q) {
      const int r = rk[q - q0];
      if (r >= 0) {
        const uint32_t bit = 1u << (r & 31);
        const bool dup = (bits[r >> 5] & bit) != 0u;
        __syncwarp();
        if (lane == 0) bits[r >> 5] |= bit;
        __syncwarp();
        if (dup) {
          err = 1;                                            // ranks are not a permutation
        } else {
          ++e;
          if (e == k) cur = warp_prev_bit(bits, S, lane);     // largest eligible rank
          else if (e > k && r < cur) cur = warp_prev_bit(bits, cur, lane);
        }
      } else if (r == -2) {
        err = 1;
      }
      if (lane == 0) out[q - q0] = e >= k ? cur : -1;
    }
    if (lane == 0 && (err || bad_sh)) raise_status(status, KVP_ERR_DEVICE_CHECK);
  }
  __syncthreads();
  for (int q = q0 + tid; q < q1; q += CT_THREADS) tau[(size_t)h * S + q] = out[q - q0];
}

}  // namespace

cudaError_t launch_topk_cutoffs(const int32_t* ranks, int n_heads, int S, int n_sink, int window,
                                int k, int32_t* tau, int* status, cudaStream_t st) {
  const int nw = (S + 31) >> 5;
  const size_t smem = ((size_t)nw + CT_THREADS + 2 * CT_CHUNK) * 4;
  cudaError_t e = cudaFuncSetAttribute(cutoff_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((S + CT_CHUNK - 1) / CT_CHUNK, n_heads);
  count_launches(1);
  cutoff_kernel<<<grid, CT_THREADS, smem, st>>>(ranks, S, n_sink, window, k, tau, status);
  return cudaGetLastError();
}

}  // namespace kvp
