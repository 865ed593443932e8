// Gather-compaction of the kept K/V rows into a dense pruned cache
// (Learning to Evict from Key-Value Cache §4.1, physical tensor compaction;
// How much KV cache can you prune, "Conclusion": kept entries copied into a
// new tensor).  Pure byte movement: every cache row (head_dim * element size
// bytes, a multiple of 16) is copied as 16-byte vectors, consecutive threads
// on consecutive vectors of the same row, so reads and writes are fully
// coalesced.  K and V of the same slot are moved by the same thread.
#include "kvp_common.cuh"
#include "kvp_launch.h"

namespace kvp {
namespace {

__device__ __forceinline__ void st_stream16(void* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

template <int VPR>   // 16-byte vectors per row
__global__ void __launch_bounds__(256) compact_kernel(const uint4* __restrict__ k,
                                                      const uint4* __restrict__ v, int R, int T,
                                                      const int32_t* __restrict__ idx,
                                                      const int32_t* __restrict__ count, int b_max,
                                                      uint4* __restrict__ ko, uint4* __restrict__ vo,
                                                      int* status) {
  const long long total = (long long)R * b_max * VPR;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += stride) {
    const int c = (int)(e % VPR);
    const long long rm = e / VPR;
    const int r = (int)(rm / b_max), m = (int)(rm % b_max);
    if (m >= count[r]) continue;
    const int src = idx[rm];
    if (src < 0 || src >= T) {
      raise_status(status, KVP_ERR_DEVICE_CHECK);
      continue;
    }
    const size_t s_off = ((size_t)r * T + src) * VPR + c;
    const uint4 a = ld_stream16(k + s_off);
    const uint4 b = ld_stream16(v + s_off);
    st_stream16(ko + rm * VPR + c, a);
    st_stream16(vo + rm * VPR + c, b);
  }
}

template <int VPR>
cudaError_t compact(const void* k, const void* v, int R, int T, const int32_t* idx,
                    const int32_t* count, int b_max, void* ko, void* vo, int* status,
                    cudaStream_t st) {
  const long long total = (long long)R * b_max * VPR;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  count_launches(1);
  compact_kernel<VPR><<<(unsigned)blocks, 256, 0, st>>>((const uint4*)k, (const uint4*)v, R, T, idx,
                                                        count, b_max, (uint4*)ko, (uint4*)vo, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compact(const void* k, const void* v, int row_bytes, int R, int T,
                           const int32_t* idx, const int32_t* count, int b_max, void* k_out,
                           void* v_out, int* status, cudaStream_t st) {
  switch (row_bytes / 16) {
    case 8: return compact<8>(k, v, R, T, idx, count, b_max, k_out, v_out, status, st);
    case 16: return compact<16>(k, v, R, T, idx, count, b_max, k_out, v_out, status, st);
    case 32: return compact<32>(k, v, R, T, idx, count, b_max, k_out, v_out, status, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvp
