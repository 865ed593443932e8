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

constexpr int RING_THREADS = 512;

// Candidate (score key, newest position first) of one slot; ~0 when the slot is protected.
__device__ __forceinline__ unsigned long long ring_key(int p, float score, int new_pos, int n_sink,
                                                       int n_recent) {
  if (p < n_sink || p > new_pos - n_recent) return ~0ull;
  return ((unsigned long long)order_key_ring(score) << 32) | (0xFFFFFFFFu - (uint32_t)p);
}

__device__ __forceinline__ void take_min(unsigned long long& best, int& slot, unsigned long long key,
                                         int m) {
  if (key < best) {
    best = key;
    slot = m;
  }
}

// All loads of a thread are issued before any comparison (the scan is latency bound: one
// row is only cap * 8 bytes), with 16-byte vectors when the row allows it; the arg-min carries
// the slot so no second pass over the positions is needed.
__global__ void __launch_bounds__(RING_THREADS) ring_insert_kernel(
    uint4* __restrict__ kc, uint4* __restrict__ vc, int32_t* __restrict__ slot_pos,
    float* __restrict__ slot_score, int32_t* __restrict__ fill, int cap, int vpr,
    const uint4* __restrict__ new_k, const uint4* __restrict__ new_v, int new_pos, int n_sink,
    int n_recent, int vec, int32_t* __restrict__ out_slot, int* status) {
  __shared__ unsigned long long best_sh[RING_THREADS / 32];
  __shared__ int slot_w[RING_THREADS / 32];
  __shared__ int slot_sh;
  const int r = blockIdx.x, tid = threadIdx.x;
  const int f = fill[r];
  int slot = -1;
  if (f < cap) {
    slot = f < 0 ? -1 : f;
  } else {
    unsigned long long best = ~0ull;
    const int32_t* pos_r = slot_pos + (size_t)r * cap;
    const float* sc_r = slot_score + (size_t)r * cap;
    if (vec) {
      const int n4 = cap >> 2;
      for (int g0 = tid; g0 < n4; g0 += 2 * RING_THREADS) {
        const int g1 = g0 + RING_THREADS;
        const int4 pa = reinterpret_cast<const int4*>(pos_r)[g0];
        const float4 sa = reinterpret_cast<const float4*>(sc_r)[g0];
        int4 pb = make_int4(-1, -1, -1, -1);
        float4 sb = make_float4(0.f, 0.f, 0.f, 0.f);
        if (g1 < n4) {
          pb = reinterpret_cast<const int4*>(pos_r)[g1];
          sb = reinterpret_cast<const float4*>(sc_r)[g1];
        }
        take_min(best, slot, ring_key(pa.x, sa.x, new_pos, n_sink, n_recent), 4 * g0);
        take_min(best, slot, ring_key(pa.y, sa.y, new_pos, n_sink, n_recent), 4 * g0 + 1);
        take_min(best, slot, ring_key(pa.z, sa.z, new_pos, n_sink, n_recent), 4 * g0 + 2);
        take_min(best, slot, ring_key(pa.w, sa.w, new_pos, n_sink, n_recent), 4 * g0 + 3);
        if (g1 < n4) {
          take_min(best, slot, ring_key(pb.x, sb.x, new_pos, n_sink, n_recent), 4 * g1);
          take_min(best, slot, ring_key(pb.y, sb.y, new_pos, n_sink, n_recent), 4 * g1 + 1);
          take_min(best, slot, ring_key(pb.z, sb.z, new_pos, n_sink, n_recent), 4 * g1 + 2);
          take_min(best, slot, ring_key(pb.w, sb.w, new_pos, n_sink, n_recent), 4 * g1 + 3);
        }
      }
    } else {
      for (int m = tid; m < cap; m += RING_THREADS)
        take_min(best, slot, ring_key(pos_r[m], sc_r[m], new_pos, n_sink, n_recent), m);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int os = __shfl_xor_sync(0xffffffffu, slot, o);
      take_min(best, slot, ob, os);
    }
    if ((tid & 31) == 0) {
      best_sh[tid >> 5] = best;
      slot_w[tid >> 5] = slot;
    }
    __syncthreads();
    if (tid < 32) {
      best = tid < RING_THREADS / 32 ? best_sh[tid] : ~0ull;
      slot = tid < RING_THREADS / 32 ? slot_w[tid] : -1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int os = __shfl_xor_sync(0xffffffffu, slot, o);
        take_min(best, slot, ob, os);
      }
      if (best == ~0ull) slot = -1;     // every slot protected
    }
  }
  if (tid == 0) slot_sh = slot;
  __syncthreads();
  slot = slot_sh;
  if (slot < 0) {
    if (tid == 0) {
      if (out_slot) out_slot[r] = -1;
      raise_status(status, KVP_ERR_DEVICE_CHECK);
    }
    return;
  }
  for (int c = tid; c < vpr; c += RING_THREADS) {
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
  const int vec = cap % 4 == 0 && ((uintptr_t)slot_pos & 15) == 0 && ((uintptr_t)slot_score & 15) == 0;
  count_launches(1);
  ring_insert_kernel<<<R, RING_THREADS, 0, st>>>((uint4*)kc, (uint4*)vc, slot_pos, slot_score, fill, cap,
                                                 row_bytes / 16, (const uint4*)new_k, (const uint4*)new_v,
                                                 new_pos, n_sink, n_recent, vec, out_slot, status);
  return cudaGetLastError();
}

}  // namespace kvp
