// fp32-FFMA tiled row-LSE and future-attention-mass passes.
//
// This is the path for float32 inputs (the tiny fp32 workload); bf16/f16
// inputs always run on the tensor cores (attn_mass_tc.cu).  Both passes use
// the same 64 x 64 register-tiled score block: 256 threads, each owning a
// 4 x 4 patch, operands staged transposed (feature-major) in shared memory so
// that every thread reads contiguous float4s.
//
//  * Row pass (KVpop, "Delayed Memory Scoring", LSE example): rows = queries,
//    columns = keys 0..i; online max / sum in base 2, one cross-lane max
//    reduction per key tile, one sum reduction at the end.
//  * Column pass (KVpop, Figure 2 "transposed attention"): rows = keys,
//    columns = queries i >= j + w of every query head of the group; each
//    thread accumulates exp2(s*log2e*scale - lse_i*log2e) of its patch rows,
//    reduced across the 16 threads of a row at the end.
#include <climits>

#include "kvp_common.cuh"
#include "kvp_launch.h"

namespace kvp {
namespace {

constexpr int TM = 64;       // rows per block
constexpr int TN = 64;       // columns per tile
constexpr int LD = TM + 4;   // padded leading dimension of the transposed tiles

// Copy rows [r0, r0 + 64) of a [S, D] matrix (row pitch `pitch` elements) into sm[d * LD + r]
// as fp32 (zeros past S).
template <typename T, int D>
__device__ __forceinline__ void load_tile_t(float* sm, const T* __restrict__ src, int r0, int S,
                                            long long pitch) {
  constexpr int V = Vec16<T>::N;   // elements per 16-byte vector
  constexpr int VPR = D / V;       // vectors per row
  for (int e = threadIdx.x; e < TM * VPR; e += blockDim.x) {
    const int r = e / VPR, c = (e % VPR) * V;
    float f[V];
    if (r0 + r < S) {
      const uint4 u = *reinterpret_cast<const uint4*>(src + (long long)(r0 + r) * pitch + c);
      Vec16<T>::unpack(u, f);
    } else {
#pragma unroll
      for (int t = 0; t < V; ++t) f[t] = 0.f;
    }
#pragma unroll
    for (int t = 0; t < V; ++t) sm[(c + t) * LD + r] = f[t];
  }
}

template <int D>
__device__ __forceinline__ void tile_dot(const float* As, const float* Bs, int ty, int tx,
                                         float acc[4][4]) {
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 8
  for (int d = 0; d < D; ++d) {
    const float4 x = *reinterpret_cast<const float4*>(As + d * LD + ty * 4);
    const float4 y = *reinterpret_cast<const float4*>(Bs + d * LD + tx * 4);
    const float xa[4] = {x.x, x.y, x.z, x.w};
    const float yb[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(xa[a], yb[b], acc[a][b]);
  }
}

__device__ __forceinline__ float row_max16(float v) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float row_sum16(float v) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ranks != null: the sparse row LSE (running top-k mask: key j is kept for query i if
// j < n_sink, j > i - window, tau_i < 0 or rank_j <= tau_i).
template <typename T, int D>
__global__ void __launch_bounds__(256) lse_simt_kernel(const T* __restrict__ q,
                                                       const T* __restrict__ k, int Hq, int Hkv,
                                                       int S, AttnShape sh, float c2,
                                                       float* __restrict__ lse,
                                                       const int32_t* __restrict__ ranks,
                                                       const int32_t* __restrict__ tau, int n_sink,
                                                       int window) {
  extern __shared__ float sm[];
  float* As = sm;
  float* Bs = sm + D * LD;
  const int i0 = blockIdx.x * TM, hq = blockIdx.y, b = blockIdx.z;
  const int G = Hq / Hkv;
  const T* qh = q + b * sh.q_sb + hq * sh.q_sh;
  const T* kh = k + b * sh.k_sb + (hq / G) * sh.k_sh;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  load_tile_t<T, D>(As, qh, i0, S, sh.q_sr);
  const int32_t* rk = ranks ? ranks + (size_t)(b * Hkv + hq / G) * S : nullptr;
  int tau_r[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int i = i0 + ty * 4 + a;
    const int tq = (rk && i < S) ? tau[(size_t)(b * Hkv + hq / G) * S + i] : -1;
    tau_r[a] = tq < 0 ? INT_MAX : tq;
  }
  float m[4], l[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) { m[a] = -INFINITY; l[a] = 0.f; }
  const int last = min(S, i0 + TM) - 1;
  for (int j0 = 0; j0 <= last; j0 += TN) {
    __syncthreads();
    load_tile_t<T, D>(Bs, kh, j0, S, sh.k_sr);
    __syncthreads();
    float acc[4][4];
    tile_dot<D>(As, Bs, ty, tx, acc);
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int i = i0 + ty * 4 + a;
      float s2[4], tmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int j = j0 + tx * 4 + c;
        bool keep = j <= i && j < S;
        if (keep && rk && j >= n_sink && j <= i - window) keep = rk[j] <= tau_r[a];
        s2[c] = keep ? acc[a][c] * c2 : -INFINITY;
        tmax = fmaxf(tmax, s2[c]);
      }
      tmax = row_max16(tmax);
      const float mn = fmaxf(m[a], tmax);
      if (mn == -INFINITY) continue;   // padding row past S: nothing visible
      float add = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) add += exp2f(s2[c] - mn);
      l[a] = l[a] * exp2f(m[a] - mn) + add;
      m[a] = mn;
    }
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const float tot = row_sum16(l[a]);
    const int i = i0 + ty * 4 + a;
    if (tx == 0 && i < S) lse[(size_t)(b * Hq + hq) * S + i] = (m[a] + log2f(tot)) * KVP_LN2;
  }
}

// per_head = 0: F[b, h, j] (group sum); per_head = 1: F[b, h*G+g, j] per query head.
template <typename T, int D>
__global__ void __launch_bounds__(256) fam_simt_kernel(const T* __restrict__ q,
                                                       const T* __restrict__ k,
                                                       const float* __restrict__ lse, int Hq,
                                                       int Hkv, int S, AttnShape sh, float c2, int w,
                                                       float* __restrict__ F, int per_head) {
  extern __shared__ float sm[];
  float* As = sm;
  float* Bs = sm + D * LD;
  float* Ls = sm + 2 * D * LD;   // lse * log2(e) of the current query tile (+inf past S)
  const int j0 = blockIdx.x * TM, hk = blockIdx.y, b = blockIdx.z;
  const int G = Hq / Hkv;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float f[4] = {0.f, 0.f, 0.f, 0.f};
  const int first = j0 + w;   // first query any key of this block receives
  if (first < S) {
    load_tile_t<T, D>(As, k + b * sh.k_sb + hk * sh.k_sh, j0, S, sh.k_sr);
    for (int g = 0; g < G; ++g) {
      const int hq = hk * G + g;
      const T* qh = q + b * sh.q_sb + hq * sh.q_sh;
      const float* lh = lse + (size_t)(b * Hq + hq) * S;
      for (int i0 = first; i0 < S; i0 += TN) {
        __syncthreads();
        load_tile_t<T, D>(Bs, qh, i0, S, sh.q_sr);
        if (threadIdx.x < TN) {
          const int i = i0 + threadIdx.x;
          Ls[threadIdx.x] = i < S ? lh[i] * KVP_LOG2E : INFINITY;
        }
        __syncthreads();
        float acc[4][4];
        tile_dot<D>(As, Bs, ty, tx, acc);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const int j = j0 + ty * 4 + a;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int i = i0 + tx * 4 + c;
            const float p = exp2f(acc[a][c] * c2 - Ls[tx * 4 + c]);
            f[a] += (i >= j + w) ? p : 0.f;
          }
        }
      }
      if (per_head) {
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const float tot = row_sum16(f[a]);
          const int j = j0 + ty * 4 + a;
          if (tx == 0 && j < S) F[(size_t)(b * Hq + hq) * S + j] = tot;
          f[a] = 0.f;
        }
      }
    }
  }
  if (per_head) {
    if (first >= S) {                        // no future queries: every head's mass is 0
      for (int e = threadIdx.x; e < G * TM; e += blockDim.x) {
        const int g = e / TM, j = j0 + e % TM;
        if (j < S) F[(size_t)(b * Hq + hk * G + g) * S + j] = 0.f;
      }
    }
    return;
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const float tot = row_sum16(f[a]);
    const int j = j0 + ty * 4 + a;
    if (tx == 0 && j < S) F[(size_t)(b * Hkv + hk) * S + j] = tot;
  }
}

// KVpop target (KVpop, "Defining Future Attention Utility" and "Alternative Aggregation
// Methods"): N_t = max(1, S - (t + w)), m_g = F_g / N_t, and per KV head either
// max_g log(eps + m_g) or log(eps + mean_g m_g); also the raw group sum of F_g.
__global__ void target_epilogue_kernel(const float* __restrict__ Fh, int Hq, int Hkv, int S, int w,
                                       float eps, int aggregate, float* __restrict__ target,
                                       float* __restrict__ F, long long total) {
  wait_prior_grid();                     // the per-head sums come from the kernel just before
  const int G = Hq / Hkv;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int j = (int)(e % S);
    const long long bh = e / S;                 // b * Hkv + h
    const int b = (int)(bh / Hkv), h = (int)(bh % Hkv);
    const float N = (float)max(1, S - (j + w));
    float sum = 0.f, best = -INFINITY;
    for (int g = 0; g < G; ++g) {
      const float fg = Fh[((size_t)b * Hq + h * G + g) * S + j];
      sum += fg;
      best = fmaxf(best, logf(eps + fg / N));
    }
    if (target) target[e] = aggregate == 0 ? best : logf(eps + sum / (N * (float)G));
    if (F) F[e] = sum;
  }
}

template <typename T, int D>
cudaError_t lse_simt(const void* q, const void* k, AttnShape s, float scale, float* lse,
                     cudaStream_t st, const SparseMask* mask) {
  const size_t smem = 2 * D * LD * sizeof(float);
  auto kern = lse_simt_kernel<T, D>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  dim3 grid((s.seq_len + TM - 1) / TM, s.h_q, s.n_batch);
  count_launches(1);
  kern<<<grid, 256, smem, st>>>((const T*)q, (const T*)k, s.h_q, s.h_kv, s.seq_len, s,
                                scale * KVP_LOG2E, lse, mask ? mask->ranks : nullptr,
                                mask ? mask->tau : nullptr, mask ? mask->n_sink : 0,
                                mask ? mask->window : 0);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t fam_simt(const void* q, const void* k, const float* lse, AttnShape s, float scale,
                     int w, float* F, cudaStream_t st, int per_head) {
  const size_t smem = (2 * D * LD + TN) * sizeof(float);
  auto kern = fam_simt_kernel<T, D>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  dim3 grid((s.seq_len + TM - 1) / TM, s.h_kv, s.n_batch);
  count_launches(1);
  kern<<<grid, 256, smem, st>>>((const T*)q, (const T*)k, lse, s.h_q, s.h_kv, s.seq_len, s,
                                scale * KVP_LOG2E, w, F, per_head);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lse_simt(const void* q, const void* k, int dtype, AttnShape s, float scale,
                            float* lse, cudaStream_t st, const SparseMask* mask) {
  if (dtype != KVP_F32) return cudaErrorInvalidValue;    // 16-bit inputs run on the tensor cores
  return s.head_dim == 128 ? lse_simt<float, 128>(q, k, s, scale, lse, st, mask)
                           : lse_simt<float, 64>(q, k, s, scale, lse, st, mask);
}

cudaError_t launch_fam_simt(const void* q, const void* k, const float* lse, int dtype, AttnShape s,
                            float scale, int w, float* F, cudaStream_t st, int per_head) {
  if (dtype != KVP_F32) return cudaErrorInvalidValue;
  return s.head_dim == 128 ? fam_simt<float, 128>(q, k, lse, s, scale, w, F, st, per_head)
                           : fam_simt<float, 64>(q, k, lse, s, scale, w, F, st, per_head);
}

cudaError_t launch_target_epilogue(const float* F_heads, int n_batch, int h_q, int h_kv, int S,
                                   int window, float eps, int aggregate, float* target, float* F,
                                   cudaStream_t st) {
  const long long total = (long long)n_batch * h_kv * S;
  long long blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  count_launches(1);
  return launch_with_pdl(target_epilogue_kernel, dim3((unsigned)blocks), dim3(256), 0, st, F_heads, h_q, h_kv, S,
                         window, eps, aggregate, target, F, total);
}

}  // namespace kvp
