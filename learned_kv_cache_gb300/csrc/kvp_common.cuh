// Device helpers shared by the kernels of libkvp (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvp.h"

#define KVP_LOG2E 1.4426950408889634f
#define KVP_LN2 0.6931471805599453f

namespace kvp {

// Programmatic dependent launch: a kernel launched with programmatic stream serialization may
// start while the previous kernel of the stream is finishing; it waits here, before its first
// access to global memory, until that kernel has completed and its writes are visible (a no-op
// when the launch was ordinary).
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Record the first device-side error in the per-device status word.
__device__ __forceinline__ void raise_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }

// Unpack a 16-byte vector of T into floats (4 for f32, 8 for 16-bit types).
template <typename T>
struct Vec16 {
  static constexpr int N = 16 / sizeof(T);
  __device__ __forceinline__ static void unpack(const uint4& u, float* f);
};
template <>
__device__ __forceinline__ void Vec16<float>::unpack(const uint4& u, float* f) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
template <>
__device__ __forceinline__ void Vec16<__nv_bfloat16>::unpack(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
template <>
__device__ __forceinline__ void Vec16<__half>::unpack(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
    float2 v = __half22float2(h);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Streaming 16-byte global load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Inclusive warp scan (int).
__device__ __forceinline__ int warp_inclusive_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Exclusive block scan for blockDim.x a multiple of 32 (<= 1024); `sh` holds 33 ints.
__device__ __forceinline__ int block_exclusive_scan(int v, int* sh, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int inc = warp_inclusive_scan(v);
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int t = lane < nw ? sh[lane] : 0;
    int ti = warp_inclusive_scan(t);
    if (lane < nw) sh[lane] = ti - t;
    if (lane == nw - 1) sh[32] = ti;
  }
  __syncthreads();
  int res = inc - v + sh[warp];
  *total = sh[32];
  __syncthreads();
  return res;
}

}  // namespace kvp
