// In-place eviction of a static (ring) decode cache.
//
// How much KV cache can you prune before quality degrades, "What we did" (the
// attention-score policy keeps the first tokens, always keeps the newest ones
// and fills the rest with the tokens that received the most attention) and
// "Conclusion" (a ring or static cache reserves a fixed region and overwrites
// old entries in place instead of selecting and copying every step).
//
// One CTA per row: while the cache is not full the new token is appended;
// otherwise a block-wide arg-min over the slots picks the lowest cumulative
// score among the slots that are neither sinks nor among the n_recent newest
// tokens (NaN first, -0.0 == +0.0, ties to the newer token), and the new
// token's K/V row is copied into it with 16-byte vectors.
#include "kvp_common.cuh"
#include "kvp_launch.h"

namespace kvp {
namespace {

__device__ __forceinline__ uint32_t order_key_ring(float x) {
  if (x != x) return 0u;
  uint32_t u = __float_as_uint(x);
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int RING_THREADS = 256;

__global__ void __launch_bounds__(RING_THREADS) ring_insert_kernel(
    uint4* __restrict__ kc, uint4* __restrict__ vc, int32_t* __restrict__ slot_pos,
    float* __restrict__ slot_score, int32_t* __restrict__ fill, int cap, int vpr,
    const uint4* __restrict__ new_k, const uint4* __restrict__ new_v, int new_pos, int n_sink,
    int n_recent, int32_t* __restrict__ out_slot, int* status) {
  __shared__ unsigned long long best_sh[RING_THREADS / 32];
  __shared__ int slot_sh;
  const int r = blockIdx.x, tid = threadIdx.x;
  const int f = fill[r];
  if (tid == 0) slot_sh = -1;
  if (f < cap) {
    if (tid == 0) slot_sh = f < 0 ? -1 : f;
  } else {
    // minimum of (score key, newest position first); positions are unique, so the winning
    // slot is found again from its position
    unsigned long long best = ~0ull;
    for (int m = tid; m < cap; m += blockDim.x) {
      const int p = slot_pos[(size_t)r * cap + m];
      if (p < n_sink || p > new_pos - n_recent) continue;
      const uint32_t sk = order_key_ring(slot_score[(size_t)r * cap + m]);
      const unsigned long long key = ((unsigned long long)sk << 32) | (0xFFFFFFFFu - (uint32_t)p);
      best = key < best ? key : best;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other < best ? other : best;
    }
    if ((tid & 31) == 0) best_sh[tid >> 5] = best;
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < RING_THREADS / 32; ++w) best = best_sh[w] < best ? best_sh[w] : best;
      best_sh[0] = best;
    }
    __syncthreads();
    best = best_sh[0];
    if (best != ~0ull) {
      const int p_best = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFu));
      for (int m = tid; m < cap; m += blockDim.x)
        if (slot_pos[(size_t)r * cap + m] == p_best) slot_sh = m;   // positions are unique
    }
  }
  __syncthreads();
  const int slot = slot_sh;
  if (slot < 0) {
    if (tid == 0) {
      if (out_slot) out_slot[r] = -1;
      raise_status(status, KVP_ERR_DEVICE_CHECK);
    }
    return;
  }
  for (int c = tid; c < vpr; c += blockDim.x) {
    kc[((size_t)r * cap + slot) * vpr + c] = new_k[(size_t)r * vpr + c];
    vc[((size_t)r * cap + slot) * vpr + c] = new_v[(size_t)r * vpr + c];
  }
  if (tid == 0) {
    slot_pos[(size_t)r * cap + slot] = new_pos;
    slot_score[(size_t)r * cap + slot] = 0.f;
    if (f < cap) fill[r] = f + 1;
    if (out_slot) out_slot[r] = slot;
  }
}

}  // namespace

cudaError_t launch_ring_insert(void* kc, void* vc, int32_t* slot_pos, float* slot_score, int32_t* fill,
                               int R, int cap, int row_bytes, const void* new_k, const void* new_v,
                               int new_pos, int n_sink, int n_recent, int32_t* out_slot, int* status,
                               cudaStream_t st) {
  count_launches(1);
  ring_insert_kernel<<<R, RING_THREADS, 0, st>>>((uint4*)kc, (uint4*)vc, slot_pos, slot_score, fill, cap,
                                                 row_bytes / 16, (const uint4*)new_k, (const uint4*)new_v,
                                                 new_pos, n_sink, n_recent, out_slot, status);
  return cudaGetLastError();
}

}  // namespace kvp
