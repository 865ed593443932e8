// Split-K decode attention over a (pruned) bf16/f16 KV cache, streamed by TMA.
//
// How much KV cache can you prune, "What we did" / "Bounded windows": one-token
// attention over the retained entries.  The kernel is HBM-bound, so it is
// built around the data movement:
//
//  * persistent grid of 2 CTAs per SM; the (row, 64-key tile) sequence of all
//    rows is cut into equal contiguous ranges, one per CTA (stream-K), so every
//    SM streams the same number of bytes whatever the row lengths;
//  * one producer warp keeps a ring of K/V tiles in flight with TMA tensor
//    loads (128-byte swizzle, so the ldmatrix reads below are conflict-free);
//  * four consumer warps each own 16 keys of a tile.  The G <= 8 query heads
//    of the GQA group share every K/V byte: the logits S^T = K Q^T and the
//    output O^T += V^T P^T are m16n8k16 products (keys or head dims in M, the
//    padded group in N) with fp32 accumulation; P is fed to the second
//    product as a hi + lo pair of 16-bit values so the weights keep ~22 bits;
//  * base-2 online softmax per query head, rescaling only when a lane group's
//    maximum grows;
//  * at the end of a row segment the four warps merge through shared memory,
//    the CTA writes one partial (max, sum, output) and the last CTA to finish a
//    row (atomic counter) merges that row's partials in CTA order
//    (deterministic) and writes the output.
// With the key mass requested, every logit is also stored ([R, T_cap, 8]) and a
// second kernel adds the group-summed probability of each key at its source
// position once the row's log-sum-exp is known.
#include <cooperative_groups.h>

#include "kvp_common.cuh"
#include "kvp_launch.h"
#include "tc_ptx.cuh"

namespace kvp {
namespace {

constexpr int DM_TILE = 64;                 // keys per pipeline stage
constexpr int DM_CWARPS = 4;                // consumer warps (16 keys of every tile each)
constexpr int DM_THREADS = 32 * (DM_CWARPS + 1);
constexpr int DM_QPAD = 8;                  // query heads of a group, padded to the MMA N

template <int D>
struct Dm {
  static constexpr int HALVES = D / 64;                     // 128-byte swizzle spans per row
  static constexpr int HALF_BYTES = DM_TILE * 128;          // one span of a 64-key tile
  static constexpr int TILE_BYTES = HALVES * HALF_BYTES;    // K (or V) of one tile
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int STAGES = D == 128 ? 2 : 4;
  static constexpr int KSTEPS = D / 16;
  static constexpr int PSTRIDE = 2 * DM_QPAD + DM_QPAD * D; // partial: m[8], l[8], o[8][D]
  static constexpr int OFF_BAR = STAGES * STAGE_BYTES;
  // Merge scratch of the four consumer warps.  It aliases the stage ring: every CTA's tile
  // range lies in one row (see decode_mma_plan), so the merge runs only after the last tile
  // has been consumed and no copy is in flight.
  static constexpr int OFF_SM = 0;
  static constexpr int OSTR = D + 4;                        // padded row of the output scratch
  static constexpr int SCRATCH = (3 * DM_CWARPS * DM_QPAD + DM_CWARPS * DM_QPAD * OSTR) * 4;
  static_assert(SCRATCH <= STAGES * STAGE_BYTES, "merge scratch must fit in the stage ring");
  static constexpr int OFF_CST = OFF_BAR + 128;             // merged state of this CTA
  static constexpr int OFF_FLAG = OFF_CST + PSTRIDE * 4;
  static constexpr int MAXC = (DM_CWARPS * DM_QPAD * D) / (2 + 2 * DM_QPAD);   // combine capacity
  static constexpr int OFF_LG = OFF_FLAG + 16;              // logits of this CTA's keys (optional)
  static constexpr int SMEM = OFF_LG + 1024;                // + alignment slack (+ logits bytes)
};

// Logits kept in shared memory for the in-kernel key mass: at most this many keys per CTA.
constexpr int DM_LG_SMEM_KEYS = 1536;

struct DmParams {
  int Hq, Hkv, G, R, T_cap, NT;
  long long total_tiles;
  int n_ctas, maxseg;
  float c2;
  const int32_t* len;
  float* partial;        // [n_ctas][maxseg][PSTRIDE]
  int* counters;         // [R], zero on entry, left zero on exit
  float* out;            // [L, Hq, D]
  float* lse2;           // [R][8] (base-2 LSE per query head, for the key mass)
  float* logits;         // [R][T_cap][8] in the workspace, or null
  int lg_smem;           // 1: the logits of a CTA's keys stay in its shared memory instead
  float* key_mass;       // [R][T_src] or null; in the cluster path accumulated in this kernel
  const int32_t* key_pos;
  int T_src;
  int* status;
  int cluster;           // > 0: the `cluster` CTAs of a row form a thread-block cluster and
                         // merge through distributed shared memory (no partials in HBM)
};

// First tile of CTA c, and the CTA that owns tile x (ranges are floor(c * total / P)).
__device__ __forceinline__ long long cta_begin(int c, const DmParams& p) {
  return (long long)c * p.total_tiles / p.n_ctas;
}
__device__ __forceinline__ int cta_of(long long x, const DmParams& p) {
  return (int)(((x + 1) * p.n_ctas - 1) / p.total_tiles);
}

__device__ __forceinline__ int row_len(const DmParams& p, int r) {
  int n = p.len[r];
  return n < 0 ? 0 : (n > p.T_cap ? p.T_cap : n);
}

template <typename T>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<__half>(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// Pack two fp32 into a 16-bit pair (lo = first), and return what was kept.
template <typename T>
__device__ __forceinline__ uint32_t pack_split(float a, float b, float& ka, float& kb);
template <>
__device__ __forceinline__ uint32_t pack_split<__half>(float a, float b, float& ka, float& kb) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  __half2 h = *reinterpret_cast<__half2*>(&r);
  ka = __low2float(h);
  kb = __high2float(h);
  return r;
}
template <>
__device__ __forceinline__ uint32_t pack_split<__nv_bfloat16>(float a, float b, float& ka, float& kb) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  ka = __uint_as_float(r << 16);
  kb = __uint_as_float(r & 0xffff0000u);
  return r;
}

// Shared address of the 16-byte chunk holding (key, d..d+7) of a swizzled tile.
template <int D>
__device__ __forceinline__ uint32_t tile_addr(uint32_t tile, int key, int d) {
  const int half = d >> 6, c = (d & 63) >> 3;
  return tile + half * Dm<D>::HALF_BYTES + key * 128 + ((c ^ (key & 7)) << 4);
}

template <typename T, int D>
__global__ void __launch_bounds__(DM_THREADS, 2)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const T* __restrict__ q, const DmParams p) {
  using C = Dm<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t bar_full = sbase + C::OFF_BAR;          // [STAGES]
  const uint32_t bar_empty = bar_full + 8 * C::STAGES;   // [STAGES]
  float* sm_m = reinterpret_cast<float*>(smem + C::OFF_SM);           // [4][8]
  float* sm_l = sm_m + DM_CWARPS * DM_QPAD;                           // [4][8]
  float* sm_w = sm_l + DM_CWARPS * DM_QPAD;                           // [4][8] merge weights
  float* sm_o = sm_w + DM_CWARPS * DM_QPAD;                           // [4][8][OSTR]
  volatile int* flags = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);  // [0] abort, [1] last
  float* cst = reinterpret_cast<float*>(smem + C::OFF_CST);          // m[8], l[8], o[8][D]
  float* sm_lg = reinterpret_cast<float*>(smem + C::OFF_LG);         // [keys of this CTA][8]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const long long x_begin = cta_begin(c, p), x_end = cta_begin(c + 1, p);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(bar_full + 8 * s, 1);
      ptx::mbar_init(bar_empty + 8 * s, DM_CWARPS);
    }
    flags[0] = 0;
    flags[1] = 0;
    ptx::fence_mbar_init();
  }
  if (threadIdx.x < DM_QPAD) {
    cst[threadIdx.x] = -INFINITY;
    cst[DM_QPAD + threadIdx.x] = 0.f;
  }
  // the cache, lengths and query may be written by the kernel just before this one
  wait_prior_grid();
  __syncthreads();

  if (warp == DM_CWARPS) {
    // ------------------------------------------------------------ producer
    if (p.key_mass && lane > 0) {
      // Warm L2 with the key-mass entries (and source positions) this CTA adds to after the
      // merge, so that the read-modify-writes at the end do not wait on DRAM.
      const int r0 = (int)(x_begin / p.NT);
      const int k_lo = (int)(x_begin - (long long)r0 * p.NT) * DM_TILE;
      int k_hi = (int)(x_end - (long long)r0 * p.NT) * DM_TILE;
      k_hi = k_hi < p.T_cap ? k_hi : p.T_cap;
      if (x_end - x_begin > 0 && (x_end - 1) / p.NT == r0) {    // a range inside one row
        for (int kk = k_lo + (lane - 1) * 32; kk < k_hi; kk += 31 * 32) {
          if (p.key_pos)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(__cvta_generic_to_global(p.key_pos + (size_t)r0 * p.T_cap + kk)));
          else
            asm volatile("prefetch.global.L2 [%0];" ::"l"(__cvta_generic_to_global(p.key_mass + (size_t)r0 * p.T_src + kk)));
        }
      }
    }
    if (lane == 0) {
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      int li = 0;
      // (row, tile) of x as running counters (one division for the start of the range)
      int rr = (int)(x_begin / p.NT), uu = (int)(x_begin - (long long)rr * p.NT);
      for (long long x = x_begin; x < x_end; ++x) {
        const int r = rr, u = uu;
        if (++uu == p.NT) {
          uu = 0;
          ++rr;
        }
        // The first tile of the range is copied without waiting for the row length (it is
        // inside the cache whatever the length); the consumers release it unread if it is
        // past the end of the row.
        if (x != x_begin && u * DM_TILE >= row_len(p, r)) continue;
        const int s = li % C::STAGES, use = li / C::STAGES;
        if (use > 0 && !ptx::mbar_wait(bar_empty + 8 * s, (use - 1) & 1, flags, p.status)) break;
        const uint32_t dst = sbase + s * C::STAGE_BYTES;
        ptx::mbar_arrive_expect_tx(bar_full + 8 * s, C::STAGE_BYTES);
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h) {
          ptx::tma_load_3d(dst + h * C::HALF_BYTES, &tmK, bar_full + 8 * s, 64 * h, u * DM_TILE, r);
          ptx::tma_load_3d(dst + C::TILE_BYTES + h * C::HALF_BYTES, &tmV, bar_full + 8 * s, 64 * h,
                           u * DM_TILE, r);
        }
        ++li;
      }
      // every copy must land before the CTA can exit
      for (int j = li - C::STAGES < 0 ? 0 : li - C::STAGES; j < li; ++j)
        ptx::mbar_wait(bar_full + 8 * (j % C::STAGES), (j / C::STAGES) & 1, flags, p.status);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int g = lane >> 2, t = lane & 3;
    uint32_t qb[C::KSTEPS][2];
    float m2[2], ls[2];
    float o[C::KSTEPS][4];
    int li = 0;
    int cur_row = -1, seg = 0;
    const int first_row = (int)(x_begin / p.NT);

    auto start_row = [&](int r) {
      const int l = r / p.Hkv, hk = r % p.Hkv;
      if (threadIdx.x == 0 && (p.len[r] < 0 || p.len[r] > p.T_cap)) raise_status(p.status, KVP_ERR_DEVICE_CHECK);
      const bool live = g < p.G;
      const T* qrow = q + ((size_t)l * p.Hq + hk * p.G + (live ? g : 0)) * D;
#pragma unroll
      for (int ks = 0; ks < C::KSTEPS; ++ks) {
        qb[ks][0] = live ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * t) : 0u;
        qb[ks][1] = live ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * t) : 0u;
      }
      m2[0] = m2[1] = -INFINITY;
      ls[0] = ls[1] = 0.f;
#pragma unroll
      for (int db = 0; db < C::KSTEPS; ++db) o[db][0] = o[db][1] = o[db][2] = o[db][3] = 0.f;
    };

    // Merge the four warps' states of row r into this CTA's partial; the last CTA of the
    // row merges all partials and writes the output.
    auto finish_row = [&](int r) {
      const int ctid = threadIdx.x;          // 0..127
      // every consumer warp is done with the stage ring before the scratch (which aliases it)
      // is written
      asm volatile("bar.sync 1, %0;" ::"r"(DM_CWARPS * 32));
      float l0 = ls[0], l1 = ls[1];
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
      }
      if (g == 0) {
        sm_m[warp * DM_QPAD + 2 * t] = m2[0];
        sm_m[warp * DM_QPAD + 2 * t + 1] = m2[1];
        sm_l[warp * DM_QPAD + 2 * t] = l0;
        sm_l[warp * DM_QPAD + 2 * t + 1] = l1;
      }
      // query-head rows padded to OSTR floats: the four t-lanes of a g write distinct banks
#pragma unroll
      for (int db = 0; db < C::KSTEPS; ++db) {
        float* ow = sm_o + warp * DM_QPAD * C::OSTR;
        ow[(2 * t) * C::OSTR + 16 * db + g] = o[db][0];
        ow[(2 * t + 1) * C::OSTR + 16 * db + g] = o[db][1];
        ow[(2 * t) * C::OSTR + 16 * db + g + 8] = o[db][2];
        ow[(2 * t + 1) * C::OSTR + 16 * db + g + 8] = o[db][3];
      }
      asm volatile("bar.sync 1, %0;" ::"r"(DM_CWARPS * 32));
      float* part = p.cluster ? cst : p.partial + ((size_t)c * p.maxseg + seg) * C::PSTRIDE;
      if (ctid < DM_QPAD) {                  // per head: the merged max, the warps' weights, the sum
        const int qh = ctid;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < DM_CWARPS; ++w) M = fmaxf(M, sm_m[w * DM_QPAD + qh]);
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < DM_CWARPS; ++w) {
          const float mw = sm_m[w * DM_QPAD + qh];
          const float wgt = (M == -INFINITY || mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
          sm_w[w * DM_QPAD + qh] = wgt;
          L = fmaf(sm_l[w * DM_QPAD + qh], wgt, L);
        }
        part[qh] = M;
        part[DM_QPAD + qh] = L;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(DM_CWARPS * 32));
      for (int e = ctid; e < p.G * D; e += DM_CWARPS * 32) {    // padded heads carry no output
        const int qh = e / D, d = e % D;
        float O = 0.f;
#pragma unroll
        for (int w = 0; w < DM_CWARPS; ++w)
          O = fmaf(sm_o[(w * DM_QPAD + qh) * C::OSTR + d], sm_w[w * DM_QPAD + qh], O);
        part[2 * DM_QPAD + qh * D + d] = O;
      }
      if (p.cluster) {                       // merged at the end through distributed shared memory
        asm volatile("bar.sync 1, %0;" ::"r"(DM_CWARPS * 32));
        ++seg;
        return;
      }
      __threadfence();
      asm volatile("bar.sync 1, %0;" ::"r"(DM_CWARPS * 32));
      const int c_lo = cta_of((long long)r * p.NT, p), c_hi = cta_of((long long)(r + 1) * p.NT - 1, p);
      if (ctid == 0) {
        const int old = atomicAdd(p.counters + r, 1);
        flags[1] = (old == c_hi - c_lo) ? 1 : 0;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(DM_CWARPS * 32));
      if (flags[1]) {
        __threadfence();
        const int l = r / p.Hkv, hk = r % p.Hkv;
        const int nc = c_hi - c_lo + 1;
        // Shared scratch (sm_o, free now): partial offsets, then per-CTA max / sum / weight.
        long long* poff = reinterpret_cast<long long*>(sm_o);              // [nc]
        float* mcs = sm_o + 2 * C::MAXC;                                  // [nc][8]
        float* lcs = mcs + C::MAXC * DM_QPAD;                             // [nc][8]
        for (int i = ctid; i < nc; i += DM_CWARPS * 32) {
          const int cc = c_lo + i;
          poff[i] = ((long long)cc * p.maxseg + (r - (int)(cta_begin(cc, p) / p.NT))) * C::PSTRIDE;
          const float4* pp = reinterpret_cast<const float4*>(p.partial + poff[i]);
          const float4 a = __ldcg(pp), b = __ldcg(pp + 1), c4 = __ldcg(pp + 2), d4 = __ldcg(pp + 3);
          float* mo = mcs + i * DM_QPAD;
          float* lo = lcs + i * DM_QPAD;
          mo[0] = a.x; mo[1] = a.y; mo[2] = a.z; mo[3] = a.w; mo[4] = b.x; mo[5] = b.y; mo[6] = b.z; mo[7] = b.w;
          lo[0] = c4.x; lo[1] = c4.y; lo[2] = c4.z; lo[3] = c4.w; lo[4] = d4.x; lo[5] = d4.y; lo[6] = d4.z; lo[7] = d4.w;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(DM_CWARPS * 32));
        if (ctid < DM_QPAD) {          // per head: max, weights, sum
          const int qh = ctid;
          float M = -INFINITY;
          for (int i = 0; i < nc; ++i) M = fmaxf(M, mcs[i * DM_QPAD + qh]);
          float L = 0.f;
          for (int i = 0; i < nc; ++i) {
            const float mw = mcs[i * DM_QPAD + qh];
            const float wgt = (mw == -INFINITY || M == -INFINITY) ? 0.f : fast_exp2(mw - M);
            mcs[i * DM_QPAD + qh] = wgt;
            L = fmaf(lcs[i * DM_QPAD + qh], wgt, L);
          }
          sm_m[qh] = M;
          sm_l[qh] = L;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(DM_CWARPS * 32));
        for (int e = ctid; e < p.G * D; e += DM_CWARPS * 32) {
          const int qh = e / D, d = e % D;
          const float L = sm_l[qh];
          float o8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          for (int i0 = 0; i0 < nc; i0 += 8) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int i = i0 + j;
              if (i < nc)
                o8[j] = fmaf(__ldcg(p.partial + poff[i] + 2 * DM_QPAD + qh * D + d), mcs[i * DM_QPAD + qh], o8[j]);
            }
          }
          const float O = ((o8[0] + o8[1]) + (o8[2] + o8[3])) + ((o8[4] + o8[5]) + (o8[6] + o8[7]));
          p.out[((size_t)l * p.Hq + hk * p.G + qh) * D + d] = L > 0.f ? O / L : 0.f;
          if (d == 0) p.lse2[r * DM_QPAD + qh] = L > 0.f ? sm_m[qh] + __log2f(L) : -INFINITY;
        }
        if (ctid == 0) p.counters[r] = 0;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(DM_CWARPS * 32));
      ++seg;
    };

    int rr = first_row, uu = (int)(x_begin - (long long)first_row * p.NT);
    for (long long x = x_begin; x < x_end; ++x) {
      const int r = rr, u = uu;
      if (++uu == p.NT) {
        uu = 0;
        ++rr;
      }
      if (r != cur_row) {
        if (cur_row >= 0) finish_row(cur_row);
        cur_row = r;
        seg = r - first_row;
        start_row(r);
      }
      const int n = row_len(p, r);
      const int key_base = u * DM_TILE;
      if (key_base >= n && x != x_begin) continue;
      const int s = li % C::STAGES;
      // On a timeout every warp keeps walking the same tiles without computing, so the
      // row-segment barriers below are still reached by all four warps.
      if (!ptx::mbar_wait(bar_full + 8 * s, (li / C::STAGES) & 1, flags, p.status)) {
        ++li;
        continue;
      }
      if (key_base >= n) {                   // the speculative first tile of an empty range
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_empty + 8 * s);
        ++li;
        continue;
      }
      const uint32_t kt = sbase + s * C::STAGE_BYTES, vt = kt + C::TILE_BYTES;
      const int kw = warp * 16;                                  // this warp's keys in the tile
      // logits S^T[16 keys x 8 heads]
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < C::KSTEPS; ++ks) {
        uint32_t a[4];
        const int j = lane >> 3;
        ldsm_x4(tile_addr<D>(kt, kw + (j & 1) * 8 + (lane & 7), 16 * ks + (j >> 1) * 8), a);
        mma16816<T>(sc, a, qb[ks][0], qb[ks][1]);
      }
      const int key0 = key_base + kw + g, key1 = key0 + 8;
      const bool v0 = key0 < n, v1 = key1 < n;
      float x0 = v0 ? sc[0] * p.c2 : -INFINITY, x1 = v0 ? sc[1] * p.c2 : -INFINITY;
      float x2 = v1 ? sc[2] * p.c2 : -INFINITY, x3 = v1 ? sc[3] * p.c2 : -INFINITY;
      if (p.lg_smem) {
        const int k0 = key0 - (int)(x_begin - (long long)r * p.NT) * DM_TILE;   // one row per CTA
        if (v0) *reinterpret_cast<float2*>(sm_lg + k0 * DM_QPAD + 2 * t) = make_float2(x0, x1);
        if (v1) *reinterpret_cast<float2*>(sm_lg + (k0 + 8) * DM_QPAD + 2 * t) = make_float2(x2, x3);
      } else if (p.logits) {
        if (v0) *reinterpret_cast<float2*>(p.logits + ((size_t)r * p.T_cap + key0) * DM_QPAD + 2 * t) = make_float2(x0, x1);
        if (v1) *reinterpret_cast<float2*>(p.logits + ((size_t)r * p.T_cap + key1) * DM_QPAD + 2 * t) = make_float2(x2, x3);
      }
      float mq0 = fmaxf(x0, x2), mq1 = fmaxf(x1, x3);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mq0 = fmaxf(mq0, __shfl_xor_sync(0xffffffffu, mq0, off));
        mq1 = fmaxf(mq1, __shfl_xor_sync(0xffffffffu, mq1, off));
      }
      const float n0 = fmaxf(m2[0], mq0), n1 = fmaxf(m2[1], mq1);
      if (__any_sync(0xffffffffu, n0 > m2[0] || n1 > m2[1])) {
        const float c0 = (n0 == -INFINITY || m2[0] == -INFINITY) ? (n0 == -INFINITY ? 1.f : 0.f) : fast_exp2(m2[0] - n0);
        const float c1 = (n1 == -INFINITY || m2[1] == -INFINITY) ? (n1 == -INFINITY ? 1.f : 0.f) : fast_exp2(m2[1] - n1);
        ls[0] *= c0;
        ls[1] *= c1;
#pragma unroll
        for (int db = 0; db < C::KSTEPS; ++db) {
          o[db][0] *= c0;
          o[db][1] *= c1;
          o[db][2] *= c0;
          o[db][3] *= c1;
        }
        m2[0] = n0;
        m2[1] = n1;
      }
      const float p0 = m2[0] == -INFINITY ? 0.f : fast_exp2(x0 - m2[0]);
      const float p1 = m2[1] == -INFINITY ? 0.f : fast_exp2(x1 - m2[1]);
      const float p2 = m2[0] == -INFINITY ? 0.f : fast_exp2(x2 - m2[0]);
      const float p3 = m2[1] == -INFINITY ? 0.f : fast_exp2(x3 - m2[1]);
      ls[0] += p0 + p2;
      ls[1] += p1 + p3;
      // P^T as B fragments (hi + lo halves): movmatrix turns the [key][head] C layout
      // into the [head][key] layout the second product reads.
      float k0, k1, k2, k3;
      const uint32_t h01 = pack_split<T>(p0, p1, k0, k1);
      const uint32_t h23 = pack_split<T>(p2, p3, k2, k3);
      float d0, d1, d2, d3;
      const uint32_t l01 = pack_split<T>(p0 - k0, p1 - k1, d0, d1);
      const uint32_t l23 = pack_split<T>(p2 - k2, p3 - k3, d2, d3);
      const uint32_t bh0 = movm_t(h01), bh1 = movm_t(h23);
      const uint32_t bl0 = movm_t(l01), bl1 = movm_t(l23);
#pragma unroll
      for (int db = 0; db < C::KSTEPS; ++db) {
        uint32_t a[4];
        const int j = lane >> 3;
        ldsm_x4_t(tile_addr<D>(vt, kw + (j >> 1) * 8 + (lane & 7), 16 * db + (j & 1) * 8), a);
        mma16816<T>(o[db], a, bh0, bh1);
        mma16816<T>(o[db], a, bl0, bl1);
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_empty + 8 * s);
      ++li;
    }
    if (cur_row >= 0) finish_row(cur_row);
  }
  if (p.cluster) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();                          // every CTA of the row has its state in shared memory
    // Every CTA of the cluster forms the row's per-head max, weights and sum from the k
    // states, then merges its own share of the G x D outputs (k independent remote loads
    // per element, all in flight together).
    const int k = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
    const int r = c / k, l = r / p.Hkv, hk = r % p.Hkv;
    __shared__ float wgt_sh[8][DM_QPAD];
    __shared__ float lsum_sh[DM_QPAD], lse_sh[DM_QPAD];
    if (warp < DM_CWARPS) {
      if (threadIdx.x < DM_QPAD) {
        const int qh = threadIdx.x;
        float mr[8], lr[8], M = -INFINITY;
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
          mr[rr] = -INFINITY;
          lr[rr] = 0.f;
          if (rr < k) {
            const float* rs = cluster.map_shared_rank(cst, rr);
            mr[rr] = rs[qh];
            lr[rr] = rs[DM_QPAD + qh];
          }
          M = fmaxf(M, mr[rr]);
        }
        float L = 0.f;
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
          const float wgt = (M == -INFINITY || mr[rr] == -INFINITY) ? 0.f : fast_exp2(mr[rr] - M);
          wgt_sh[rr][qh] = wgt;
          L = fmaf(lr[rr], wgt, L);
        }
        lsum_sh[qh] = L;
        lse_sh[qh] = L > 0.f ? M + __log2f(L) : -INFINITY;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(DM_CWARPS * 32));
      const float* ro[8];
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) ro[rr] = cluster.map_shared_rank(cst, rr < k ? rr : 0) + 2 * DM_QPAD;
      const int E = p.G * D, e_lo = rank * E / k, e_hi = (rank + 1) * E / k;
      for (int e = e_lo + threadIdx.x; e < e_hi; e += DM_CWARPS * 32) {
        const int qh = e / D;
        float ov[8];
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) ov[rr] = rr < k ? ro[rr][e] : 0.f;
        float O = 0.f;
#pragma unroll
        for (int rr = 0; rr < 8; ++rr)
          if (rr < k) O = fmaf(ov[rr], wgt_sh[rr][qh], O);
        const float L = lsum_sh[qh];
        p.out[((size_t)l * p.Hq + hk * p.G) * D + e] = L > 0.f ? O / L : 0.f;
      }
    }
    // Remote reads are finished (their values are used above); the barrier that keeps every
    // CTA's shared memory alive until then is arrived at without release semantics, so the
    // output stores need not drain first, and the key mass below overlaps the wait.
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    if (p.key_mass && warp < DM_CWARPS) {
      // Key mass of this CTA's own keys: sum_g exp2(logit - lse2) for each key it scored.
      const int n = row_len(p, r);
      const int key_lo = (int)(x_begin - (long long)r * p.NT) * DM_TILE;
      int key_hi = (int)(x_end - (long long)r * p.NT) * DM_TILE;
      key_hi = key_hi < n ? key_hi : n;
      float lse_r[DM_QPAD];
#pragma unroll
      for (int qh = 0; qh < DM_QPAD; ++qh) lse_r[qh] = qh < p.G ? lse_sh[qh] : INFINITY;
      const int nk = key_hi - key_lo;
      auto key_sum = [&](int j) -> float {          // sum_g exp2(logit - lse2) of key key_lo + j
        const float* lg = p.lg_smem ? sm_lg + j * DM_QPAD
                                    : p.logits + ((size_t)r * p.T_cap + key_lo + j) * DM_QPAD;
        const float4 a = *reinterpret_cast<const float4*>(lg);
        const float4 b = *reinterpret_cast<const float4*>(lg + 4);
        return ((fast_exp2(a.x - lse_r[0]) + fast_exp2(a.y - lse_r[1])) +
                (fast_exp2(a.z - lse_r[2]) + fast_exp2(a.w - lse_r[3]))) +
               ((fast_exp2(b.x - lse_r[4]) + fast_exp2(b.y - lse_r[5])) +
                (fast_exp2(b.z - lse_r[6]) + fast_exp2(b.w - lse_r[7])));
      };
      if (!p.key_pos && (p.T_src & 3) == 0 && (reinterpret_cast<uintptr_t>(p.key_mass) & 15) == 0) {
        // Identity positions: this CTA alone owns its keys' entries, so a plain vector
        // read-modify-write of four consecutive keys per thread replaces the atomics.
        float* km = p.key_mass + (size_t)r * p.T_src + key_lo;
        constexpr int STEP = 4 * DM_CWARPS * 32;
        for (int j0 = 4 * threadIdx.x; j0 < nk; j0 += 2 * STEP) {
          const int j1 = j0 + STEP;
          float4 o0 = make_float4(0.f, 0.f, 0.f, 0.f), o1 = o0;
          if (j0 + 3 < nk) o0 = *reinterpret_cast<const float4*>(km + j0);
          if (j1 + 3 < nk) o1 = *reinterpret_cast<const float4*>(km + j1);
          float m0[4], m1[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            m0[u] = j0 + u < nk ? key_sum(j0 + u) : 0.f;
            m1[u] = j1 + u < nk ? key_sum(j1 + u) : 0.f;
          }
          if (j0 + 3 < nk) {
            o0.x += m0[0]; o0.y += m0[1]; o0.z += m0[2]; o0.w += m0[3];
            *reinterpret_cast<float4*>(km + j0) = o0;
          } else {
            for (int u = 0; u < 4; ++u)
              if (j0 + u < nk) km[j0 + u] += m0[u];
          }
          if (j1 + 3 < nk) {
            o1.x += m1[0]; o1.y += m1[1]; o1.z += m1[2]; o1.w += m1[3];
            *reinterpret_cast<float4*>(km + j1) = o1;
          } else {
            for (int u = 0; u < 4; ++u)
              if (j1 + u < nk) km[j1 + u] += m1[u];
          }
        }
      } else {
        for (int j = threadIdx.x; j < nk; j += DM_CWARPS * 32) {
          const float pm = key_sum(j);
          const int pos = p.key_pos ? p.key_pos[(size_t)r * p.T_cap + key_lo + j] : key_lo + j;
          if (pos < 0 || pos >= p.T_src) {
            raise_status(p.status, KVP_ERR_DEVICE_CHECK);
            continue;
          }
          atomicAdd(p.key_mass + (size_t)r * p.T_src + pos, pm);
        }
      }
    }
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  } else {
    __syncthreads();
  }
}

// key_mass[r, pos(m)] (+)= sum_g exp2(logit[r, m, g] - lse2[r, g]) for m < len[r].
__global__ void key_mass_mma_kernel(int G, int R, int T_cap, const int32_t* __restrict__ len,
                                    const float* __restrict__ logits, const float* __restrict__ lse2,
                                    const int32_t* __restrict__ key_pos, int T_src,
                                    float* __restrict__ key_mass, int* status) {
  const long long total = (long long)R * T_cap;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(e / T_cap), m = (int)(e % T_cap);
    int n = len[r];
    n = n < 0 ? 0 : (n > T_cap ? T_cap : n);
    if (m >= n) continue;
    const float4* lg = reinterpret_cast<const float4*>(logits + e * DM_QPAD);
    const float4 a = lg[0], b = lg[1];
    const float s[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float pm = 0.f;
    for (int qh = 0; qh < G; ++qh) pm += fast_exp2(s[qh] - lse2[r * DM_QPAD + qh]);
    const int pos = key_pos ? key_pos[e] : m;
    if (pos < 0 || pos >= T_src) {
      raise_status(status, KVP_ERR_DEVICE_CHECK);
      continue;
    }
    atomicAdd(key_mass + (size_t)r * T_src + pos, pm);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool make_cache_tmap(CUtensorMap* m, const void* base, int dtype, int R, int T_cap, int D) {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult qres;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qres) !=
            cudaSuccess ||
        qres != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T_cap, (cuuint64_t)R};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)T_cap * D * 2};
  cuuint32_t box[3] = {64, DM_TILE, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt =
      dtype == KVP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

template <typename T, int D>
cudaError_t run(const void* q, const void* kc, const void* vc, int dtype, int n_layers, int h_q,
                int h_kv, int T_cap, const int32_t* len, float scale, float* out, float* key_mass,
                const int32_t* key_pos, int T_src, int accumulate, const DecodePlan& plan, void* ws,
                int* status, cudaStream_t st) {
  CUtensorMap tk, tv;
  if (!make_cache_tmap(&tk, kc, dtype, plan.R, T_cap, D) || !make_cache_tmap(&tv, vc, dtype, plan.R, T_cap, D))
    return cudaErrorInvalidValue;
  char* base = (char*)ws;
  DmParams p{};
  p.Hq = h_q;
  p.Hkv = h_kv;
  p.G = h_q / h_kv;
  p.R = plan.R;
  p.T_cap = T_cap;
  p.NT = plan.nt;
  p.total_tiles = (long long)plan.R * plan.nt;
  p.n_ctas = plan.n_ctas;
  p.maxseg = plan.maxseg;
  p.c2 = scale * KVP_LOG2E;
  p.len = len;
  p.partial = (float*)base;
  p.counters = (int*)(base + plan.mma_partial_bytes);
  p.lse2 = (float*)(base + plan.mma_partial_bytes + plan.counter_bytes);
  p.logits = key_mass ? (float*)(base + plan.mma_partial_bytes + plan.counter_bytes + plan.mma_lse_bytes)
                      : nullptr;
  p.out = out;
  p.status = status;
  const int k = plan.n_ctas / plan.R;
  p.cluster = k <= 8 ? k : 0;
  // cluster path: the key mass is added inside the decode kernel (logits in shared memory when
  // a CTA's keys fit, else in the workspace); otherwise a second kernel adds it
  p.lg_smem = key_mass && p.cluster && plan.lg_smem_keys > 0;
  if (p.lg_smem) p.logits = nullptr;
  p.key_mass = p.cluster ? key_mass : nullptr;
  p.key_pos = key_pos;
  p.T_src = T_src;
  cudaError_t e = cudaSuccess;
  if (key_mass && !accumulate) {
    e = cudaMemsetAsync(key_mass, 0, (size_t)plan.R * T_src * sizeof(float), st);
    if (e != cudaSuccess) return e;
  }
  if (!p.cluster) {
    e = cudaMemsetAsync(p.counters, 0, plan.counter_bytes, st);
    if (e != cudaSuccess) return e;
  }
  const int smem_bytes = Dm<D>::SMEM + (p.lg_smem ? plan.lg_smem_keys * DM_QPAD * (int)sizeof(float) : 0);
  auto kern = decode_mma_kernel<T, D>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)plan.n_ctas);
  cfg.blockDim = dim3(DM_THREADS);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.cluster ? p.cluster : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attribute();
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  count_launches(1);
  e = cudaLaunchKernelEx(&cfg, kern, tk, tv, (const T*)q, p);
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess || !key_mass || p.cluster) return e;
  const long long total = (long long)plan.R * T_cap;
  long long blocks = (total + 255) / 256;
  if (blocks > 8192) blocks = 8192;
  count_launches(1);
  key_mass_mma_kernel<<<(unsigned)blocks, 256, 0, st>>>(p.G, plan.R, T_cap, len, p.logits, p.lse2, key_pos,
                                                       T_src, key_mass, status);
  return cudaGetLastError();
}

}  // namespace

void decode_mma_plan(DecodePlan& p, int head_dim, int T_cap, int with_key_mass) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  p.nt = (T_cap + DM_TILE - 1) / DM_TILE;
  // k CTAs per row (n_ctas = R * k): every CTA's tile range then lies inside one row, about
  // 2 CTAs per SM in total, and at least 4 tiles per CTA (8 measured slower on short rows:
  // 8 rows x 2048 keys 12.2 -> 10.2 us, 56 rows x 512 keys 14.3 -> 12.3 us for one launch).
  long long k = (2LL * sms) / p.R;
  if (k > p.nt / 4) k = p.nt / 4;
  if (k > 112) k = 112;                 // contributors one combine can hold in shared memory
  if (k < 1) k = 1;
  p.n_ctas = (int)(p.R * k);
  p.maxseg = 1;
  const int pstride = 2 * DM_QPAD + DM_QPAD * head_dim;
  p.mma_partial_bytes = align256((size_t)p.n_ctas * p.maxseg * pstride * sizeof(float));
  p.counter_bytes = align256((size_t)p.R * sizeof(int));
  p.mma_lse_bytes = align256((size_t)p.R * DM_QPAD * sizeof(float));
  // logits of the in-kernel key mass: in shared memory when every CTA of a clustered row
  // (k <= 8) scores at most DM_LG_SMEM_KEYS keys, else in the workspace
  const long long keys_per_cta = (p.nt + k - 1) / k * DM_TILE;
  p.lg_smem_keys = (with_key_mass && k <= 8 && keys_per_cta <= DM_LG_SMEM_KEYS) ? (int)keys_per_cta : 0;
  p.mma_logit_bytes = with_key_mass && !p.lg_smem_keys
                          ? align256((size_t)p.R * T_cap * DM_QPAD * sizeof(float)) : 0;
  p.mma_total_bytes = p.mma_partial_bytes + p.counter_bytes + p.mma_lse_bytes + p.mma_logit_bytes;
}

cudaError_t launch_decode_mma(const void* q, const void* kc, const void* vc, int dtype, int n_layers,
                              int h_q, int h_kv, int head_dim, int T_cap, const int32_t* len,
                              float scale, float* out, float* key_mass, const int32_t* key_pos,
                              int T_src, int accumulate, const DecodePlan& plan, void* ws,
                              int* status, cudaStream_t st) {
#define KVP_DM(TT, DD)                                                                             \
  return run<TT, DD>(q, kc, vc, dtype, n_layers, h_q, h_kv, T_cap, len, scale, out, key_mass, key_pos, \
                     T_src, accumulate, plan, ws, status, st)
  if (dtype == KVP_BF16) {
    if (head_dim == 128) KVP_DM(__nv_bfloat16, 128);
    KVP_DM(__nv_bfloat16, 64);
  }
  if (head_dim == 128) KVP_DM(__half, 128);
  KVP_DM(__half, 64);
#undef KVP_DM
}

}  // namespace kvp
