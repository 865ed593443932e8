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
  wait_prior_grid();                     // indices and counts may come from the kernel just before
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, compact_kernel<VPR>, (const uint4*)k, (const uint4*)v, R, T, idx,
                                     count, b_max, (uint4*)ko, (uint4*)vo, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Chunked prefill-compress (Learning to Evict from Key-Value Cache §4, §4.1: each chunk of a
// long prefill is appended and the cache compressed back to the budget with physical
// compaction): kept index m of row r refers to the concatenation [cache ; chunk]; K/V rows are
// copied as above and the thread of vector 0 also moves the slot's score and source position.
template <int VPR>
__global__ void __launch_bounds__(256) chunk_compact_kernel(const ChunkSrc src, int R,
                                                            const int32_t* __restrict__ idx,
                                                            const int32_t* __restrict__ count,
                                                            int b_max, uint4* __restrict__ ko,
                                                            uint4* __restrict__ vo,
                                                            float* __restrict__ so,
                                                            int32_t* __restrict__ po, int out_cap,
                                                            int* status) {
  const long long total = (long long)R * b_max * VPR;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const int T = src.n_in + src.C;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += stride) {
    const int c = (int)(e % VPR);
    const long long rm = e / VPR;
    const int r = (int)(rm / b_max), m = (int)(rm % b_max);
    if (m >= count[r]) continue;
    const int j = idx[rm];
    if (j < 0 || j >= T) {
      raise_status(status, KVP_ERR_DEVICE_CHECK);
      continue;
    }
    const uint4 *ks, *vs;
    size_t s_off;
    if (j < src.n_in) {
      ks = reinterpret_cast<const uint4*>(src.cache_k);
      vs = reinterpret_cast<const uint4*>(src.cache_v);
      s_off = ((size_t)r * src.cap_in + j) * VPR + c;
    } else {
      ks = reinterpret_cast<const uint4*>(src.chunk_k);
      vs = reinterpret_cast<const uint4*>(src.chunk_v);
      s_off = ((size_t)r * src.C + (j - src.n_in)) * VPR + c;
    }
    const uint4 a = ld_stream16(ks + s_off);
    const uint4 b = ld_stream16(vs + s_off);
    const size_t d_off = ((size_t)r * out_cap + m) * VPR + c;
    st_stream16(ko + d_off, a);
    st_stream16(vo + d_off, b);
    if (c == 0) {
      const bool in_cache = j < src.n_in;
      so[(size_t)r * out_cap + m] = in_cache ? src.cache_score[(size_t)r * src.cap_in + j]
                                             : src.chunk_score[(size_t)r * src.C + (j - src.n_in)];
      po[(size_t)r * out_cap + m] = in_cache ? src.cache_pos[(size_t)r * src.cap_in + j]
                                             : src.pos0 + (j - src.n_in);
    }
  }
}

template <int VPR>
cudaError_t chunk_compact(const ChunkSrc& src, int R, const int32_t* idx, const int32_t* count,
                          int b_max, void* ko, void* vo, float* so, int32_t* po, int out_cap,
                          int* status, cudaStream_t st) {
  const long long total = (long long)R * b_max * VPR;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  count_launches(1);
  chunk_compact_kernel<VPR><<<(unsigned)blocks, 256, 0, st>>>(src, R, idx, count, b_max, (uint4*)ko,
                                                              (uint4*)vo, so, po, out_cap, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_compact(const ChunkSrc& src, int row_bytes, int R, const int32_t* idx,
                                 const int32_t* count, int b_max, void* out_k, void* out_v,
                                 float* out_score, int32_t* out_pos, int out_cap, int* status,
                                 cudaStream_t st) {
  switch (row_bytes / 16) {
    case 8: return chunk_compact<8>(src, R, idx, count, b_max, out_k, out_v, out_score, out_pos, out_cap, status, st);
    case 16: return chunk_compact<16>(src, R, idx, count, b_max, out_k, out_v, out_score, out_pos, out_cap, status, st);
    case 32: return chunk_compact<32>(src, R, idx, count, b_max, out_k, out_v, out_score, out_pos, out_cap, status, st);
    default: return cudaErrorInvalidValue;
  }
}

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
