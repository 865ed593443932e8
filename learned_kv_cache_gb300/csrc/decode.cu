// Split-K single-token decode attention over a (pruned) KV cache.
//
// How much KV cache can you prune, "What we did" / "Bounded windows": each
// decode step runs one-token attention over the retained entries only.  The
// work is HBM streaming of K and V, so the kernel is laid out for bandwidth:
//
//  * grid = (key chunk, row r = (layer, KV head)); every CTA streams one
//    chunk of its row once and serves all G query heads of the group from it;
//  * each key row (head_dim * element bytes) is read by a group of lanes with
//    16-byte loads, so a warp consumes whole 128-byte lines per instruction;
//    the partial dot products are reduced across the lane group with
//    butterfly shuffles;
//  * softmax state (running max, sum, unnormalised output) lives in base 2,
//    rescaled only when a new maximum appears;
//  * per-CTA partials (max, sum, output) go to the workspace; a combine
//    kernel merges the chunks of a row in fixed order (deterministic).
// The optional key-mass output (the cumulative past-attention score) stores
// each logit in the workspace and, once the row's log-sum-exp is known,
// adds the group-summed probability of every retained key at its source
// position.
#include <mutex>

#include "kvp_common.cuh"
#include "kvp_launch.h"

namespace kvp {
namespace {

// Scratch of kvp_decode_attn_noalloc: the split-K partials live here instead
// of in a caller-provided workspace.  Every GPU that loads the library keeps
// this array for the life of the process; all calls on a device share it.
static __device__ __align__(256) unsigned char g_decode_noalloc_scratch[KVP_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoallocMaxDevices] = {nullptr};
void* g_noalloc_ctx[kNoallocMaxDevices] = {nullptr};   // context each cached address belongs to

constexpr int MAXG = 8;
constexpr int DEC_WARPS = 4;
constexpr int DEC_UNROLL = 4;

template <typename T, int D>
struct DecodeCfg {
  static constexpr int EV = 16 / sizeof(T);      // elements per 16-byte vector
  static constexpr int LPK = D / EV;             // lanes per key row
  static constexpr int KPW = 32 / LPK;           // keys per warp step
  static constexpr int NS = DEC_WARPS * KPW;     // independent softmax states per CTA
};

template <typename T, int D>
__global__ void __launch_bounds__(DEC_WARPS * 32) decode_split_kernel(
    const T* __restrict__ q, const T* __restrict__ kc, const T* __restrict__ vc, int Hq, int Hkv,
    int T_cap, const int32_t* __restrict__ len, float c2, int chunk, int n_chunks,
    float* __restrict__ partial, float* __restrict__ logits, int* status) {
  using C = DecodeCfg<T, D>;
  constexpr int EV = C::EV, LPK = C::LPK, KPW = C::KPW, NS = C::NS;
  __shared__ float st_m[NS][MAXG], st_l[NS][MAXG];
  __shared__ float st_o[NS][MAXG][D];

  const int c = blockIdx.x, r = blockIdx.y;
  const int G = Hq / Hkv, l = r / Hkv, hk = r % Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane / LPK, dl = lane % LPK;
  int n = len[r];
  if (n < 0 || n > T_cap) {
    if (threadIdx.x == 0 && c == 0) raise_status(status, KVP_ERR_DEVICE_CHECK);
    n = n < 0 ? 0 : T_cap;
  }
  const int m_lo = c * chunk, m_hi = min(n, m_lo + chunk);

  float qf[MAXG][EV];
#pragma unroll
  for (int g = 0; g < MAXG; ++g) {
    if (g < G) {
      const uint4 u = *reinterpret_cast<const uint4*>(q + ((size_t)l * Hq + hk * G + g) * D + dl * EV);
      Vec16<T>::unpack(u, qf[g]);
#pragma unroll
      for (int t = 0; t < EV; ++t) qf[g][t] *= c2;
    }
  }
  float mx[MAXG], sm[MAXG], o[MAXG][EV];
#pragma unroll
  for (int g = 0; g < MAXG; ++g) {
    mx[g] = -INFINITY;
    sm[g] = 0.f;
#pragma unroll
    for (int t = 0; t < EV; ++t) o[g][t] = 0.f;
  }

  const T* krow = kc + (size_t)r * T_cap * D + dl * EV;
  const T* vrow = vc + (size_t)r * T_cap * D + dl * EV;
  constexpr int STEP = DEC_WARPS * KPW;
  for (int mb = m_lo + warp * KPW + sub; mb - sub < m_hi; mb += STEP * DEC_UNROLL) {
    uint4 ku[DEC_UNROLL], vu[DEC_UNROLL];
    bool valid[DEC_UNROLL];
#pragma unroll
    for (int u = 0; u < DEC_UNROLL; ++u) {
      const int m = mb + u * STEP;
      valid[u] = m < m_hi;
      ku[u] = valid[u] ? ld_stream16(krow + (size_t)m * D) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < DEC_UNROLL; ++u) {
      const int m = mb + u * STEP;
      vu[u] = valid[u] ? ld_stream16(vrow + (size_t)m * D) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < DEC_UNROLL; ++u) {
      const int m = mb + u * STEP;
      float kf[EV], vf[EV];
      Vec16<T>::unpack(ku[u], kf);
      Vec16<T>::unpack(vu[u], vf);
#pragma unroll
      for (int g = 0; g < MAXG; ++g) {
        if (g >= G) break;
        float s = 0.f;
#pragma unroll
        for (int t = 0; t < EV; ++t) s = fmaf(qf[g][t], kf[t], s);
#pragma unroll
        for (int off = LPK / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (!valid[u]) continue;
        if (logits && dl == 0) logits[((size_t)r * G + g) * T_cap + m] = s;
        if (s > mx[g]) {
          const float corr = fast_exp2(mx[g] - s);
          sm[g] *= corr;
#pragma unroll
          for (int t = 0; t < EV; ++t) o[g][t] *= corr;
          mx[g] = s;
        }
        const float p = fast_exp2(s - mx[g]);
        sm[g] += p;
#pragma unroll
        for (int t = 0; t < EV; ++t) o[g][t] = fmaf(p, vf[t], o[g][t]);
      }
    }
  }
  // Merge the NS per-(warp, lane group) states of this CTA.
  const int si = warp * KPW + sub;
#pragma unroll
  for (int g = 0; g < MAXG; ++g) {
    if (g >= G) break;
    if (dl == 0) { st_m[si][g] = mx[g]; st_l[si][g] = sm[g]; }
#pragma unroll
    for (int t = 0; t < EV; ++t) st_o[si][g][dl * EV + t] = o[g][t];
  }
  __syncthreads();
  float* part = partial + ((size_t)r * n_chunks + c) * G * (D + 2);
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int g = e / D, d = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < NS; ++s) M = fmaxf(M, st_m[s][g]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        const float wgt = fast_exp2(st_m[s][g] - M);
        L = fmaf(st_l[s][g], wgt, L);
        O = fmaf(st_o[s][g][d], wgt, O);
      }
    }
    if (d == 0) { part[g * (D + 2)] = M; part[g * (D + 2) + 1] = L; }
    part[g * (D + 2) + 2 + d] = O;
  }
}

template <typename T, int D>
__global__ void decode_combine_kernel(int Hq, int Hkv, int n_chunks, const float* __restrict__ partial,
                                      float* __restrict__ out, float* __restrict__ lse2) {
  const int r = blockIdx.x;
  const int G = Hq / Hkv, l = r / Hkv, hk = r % Hkv;
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int g = e / D, d = e % D;
    const float* p = partial + (size_t)r * n_chunks * G * (D + 2) + g * (D + 2);
    const size_t cs = (size_t)G * (D + 2);
    float M = -INFINITY;
    for (int c = 0; c < n_chunks; ++c) M = fmaxf(M, p[c * cs]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int c = 0; c < n_chunks; ++c) {
        const float wgt = fast_exp2(p[c * cs] - M);
        L = fmaf(p[c * cs + 1], wgt, L);
        O = fmaf(p[c * cs + 2 + d], wgt, O);
      }
    }
    out[((size_t)l * Hq + hk * G + g) * D + d] = L > 0.f ? O / L : 0.f;
    if (d == 0) lse2[r * G + g] = L > 0.f ? M + log2f(L) : -INFINITY;
  }
}

__global__ void key_mass_kernel(int Hq, int Hkv, int R, int T_cap, const int32_t* __restrict__ len,
                                const float* __restrict__ logits, const float* __restrict__ lse2,
                                const int32_t* __restrict__ key_pos, int T_src,
                                float* __restrict__ key_mass, int* status) {
  const int G = Hq / Hkv;
  const long long total = (long long)R * T_cap;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(e / T_cap), m = (int)(e % T_cap);
    const int n = min(max(len[r], 0), T_cap);
    if (m >= n) continue;
    float p = 0.f;
    for (int g = 0; g < G; ++g)
      p += fast_exp2(logits[((size_t)r * G + g) * T_cap + m] - lse2[r * G + g]);
    const int pos = key_pos ? key_pos[e] : m;
    if (pos < 0 || pos >= T_src) {
      raise_status(status, KVP_ERR_DEVICE_CHECK);
      continue;
    }
    atomicAdd(key_mass + (size_t)r * T_src + pos, p);
  }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

template <typename T, int D>
cudaError_t decode(const void* q, const void* kc, const void* vc, int n_layers, int h_q, int h_kv,
                   int T_cap, const int32_t* len, float scale, float* out, float* key_mass,
                   const int32_t* key_pos, int T_src, int accumulate, const DecodePlan& plan,
                   void* ws, int* status, cudaStream_t st) {
  char* base = (char*)ws;
  float* partial = (float*)base;
  float* lse2 = (float*)(base + plan.partial_bytes);
  float* logits = key_mass ? (float*)(base + plan.partial_bytes + plan.lse_bytes) : nullptr;
  dim3 grid(plan.n_chunks, plan.R);
  count_launches(1);
  decode_split_kernel<T, D><<<grid, DEC_WARPS * 32, 0, st>>>(
      (const T*)q, (const T*)kc, (const T*)vc, h_q, h_kv, T_cap, len, scale * KVP_LOG2E,
      plan.chunk, plan.n_chunks, partial, logits, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int G = h_q / h_kv;
  int thr = ((G * D + 31) / 32) * 32;
  if (thr > 1024) thr = 1024;
  count_launches(1);
  decode_combine_kernel<T, D><<<plan.R, thr, 0, st>>>(h_q, h_kv, plan.n_chunks, partial, out, lse2);
  e = cudaGetLastError();
  if (e != cudaSuccess || !key_mass) return e;
  if (!accumulate) {
    e = cudaMemsetAsync(key_mass, 0, (size_t)plan.R * T_src * sizeof(float), st);
    if (e != cudaSuccess) return e;
  }
  const long long total = (long long)plan.R * T_cap;
  long long blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  count_launches(1);
  key_mass_kernel<<<(unsigned)blocks, 256, 0, st>>>(h_q, h_kv, plan.R, T_cap, len, logits, lse2,
                                                   key_pos, T_src, key_mass, status);
  return cudaGetLastError();
}

}  // namespace

DecodePlan decode_plan(int n_layers, int h_q, int h_kv, int head_dim, int T_cap, int with_key_mass) {
  DecodePlan p;
  p.R = n_layers * h_kv;
  p.G = h_q / h_kv;
  long long target = ((long long)T_cap * p.R + 1215) / 1216;   // ~8 CTAs per SM over 152 SMs
  long long ch = ((target + 63) / 64) * 64;
  if (ch < 64) ch = 64;
  if (ch > 4096) ch = 4096;
  p.chunk = (int)ch;
  p.n_chunks = (int)((T_cap + ch - 1) / ch);
  if (p.n_chunks < 1) p.n_chunks = 1;
  p.partial_bytes = align256((size_t)p.R * p.n_chunks * p.G * (head_dim + 2) * sizeof(float));
  p.lse_bytes = align256((size_t)p.R * p.G * sizeof(float));
  p.logit_bytes = with_key_mass ? align256((size_t)p.R * p.G * T_cap * sizeof(float)) : 0;
  p.simt_total_bytes = p.partial_bytes + p.lse_bytes + p.logit_bytes;
  decode_mma_plan(p, head_dim, T_cap, with_key_mass);
  p.total_bytes = p.simt_total_bytes > p.mma_total_bytes ? p.simt_total_bytes : p.mma_total_bytes;
  return p;
}

// Device address of the static decode scratch on the current device.  In host
// code the array's name only stands in for the symbol, so the address is
// looked up with cudaGetSymbolAddress, with that device current, and cached
// per device together with the CUDA context it belongs to: a new context on
// the device (after cudaDeviceReset) loads the module again, possibly at
// another address, and the address is then looked up again.
bool decode_noalloc_scratch_ready() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoallocMaxDevices) return false;
  void* ctx = current_cu_context();
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  return g_noalloc_ptr[dev] != nullptr && g_noalloc_ctx[dev] == ctx;
}

cudaError_t decode_noalloc_scratch(void** ptr, size_t* bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoallocMaxDevices) return cudaErrorInvalidDevice;
  void* ctx = current_cu_context();
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev] || g_noalloc_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = p;
    g_noalloc_ctx[dev] = ctx;
  }
  *ptr = g_noalloc_ptr[dev];
  *bytes = sizeof(g_decode_noalloc_scratch);
  return cudaSuccess;
}

cudaError_t launch_decode(const void* q, const void* kc, const void* vc, int dtype, int n_layers,
                          int h_q, int h_kv, int head_dim, int T_cap, const int32_t* len,
                          float scale, float* out, float* key_mass, const int32_t* key_pos,
                          int T_src, int accumulate, const DecodePlan& plan, void* ws,
                          int* status, cudaStream_t st) {
#define KVP_DEC(TT, DD)                                                                            \
  return decode<TT, DD>(q, kc, vc, n_layers, h_q, h_kv, T_cap, len, scale, out, key_mass, key_pos, \
                        T_src, accumulate, plan, ws, status, st)
  if (dtype != KVP_F32)
    return launch_decode_mma(q, kc, vc, dtype, n_layers, h_q, h_kv, head_dim, T_cap, len, scale, out,
                             key_mass, key_pos, T_src, accumulate, plan, ws, status, st);
  if (head_dim == 128) KVP_DEC(float, 128);
  KVP_DEC(float, 64);
#undef KVP_DEC
}

}  // namespace kvp
