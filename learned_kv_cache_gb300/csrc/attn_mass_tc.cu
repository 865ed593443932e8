// Tensor-core row-LSE and future-attention-mass passes (sm_103a: tcgen05 MMA
// with TMEM accumulators, operands staged by TMA in 128-byte-swizzled shared
// memory).
//
// Both passes are the same contraction, S = A * B^T with A a fixed 128-row
// tile of the CTA and B a stream of 128-row tiles, followed by a fused
// per-row softmax epilogue that reads the fp32 scores straight from TMEM:
//
//  * row LSE (KVpop, "Delayed Memory Scoring", LSE worked example): A = a
//    query tile, B = the key tiles 0..qt (causal); each TMEM lane is one query
//    row; online max / sum in base 2; the diagonal tile is masked j <= i.
//  * sparse row LSE (KVpop, "Efficient Online Pruning" and "Delayed Memory
//    Scoring": the student's sparse log-normalisers): the row-LSE pass with the
//    running top-k mask applied per element before the exp -- sinks, the
//    protected window and the eligible keys whose static rank is within the
//    query's cutoff.
//  * future-attention mass (KVpop, Figure 2, transposed attention): roles
//    swapped, A = a key tile, B = the query tiles i >= j + w of every query
//    head of the GQA group; each TMEM lane is one key row and simply
//    accumulates exp2(s*log2e*scale - lse_i*log2e) over its columns, so the
//    column sums of the attention matrix become per-thread row sums with no
//    atomics; only the first query tile (the window diagonal) is masked
//    i >= j + w; queries past S get lse = +inf (weight 0).
//
// CTA layout (320 threads, 2 CTAs per SM): warps 0-7 epilogue (warp w reads
// TMEM lanes 32*(w%4).., column half w/4 of each tile), warp 8 TMA producer,
// warp 9 TMEM allocator + MMA issuer (one elected thread).  Shared memory:
// A tile (32 KB) + 2 B stages (2 x 32 KB); TMEM: 2 accumulators of 128 fp32
// columns so the MMA of tile t+1 overlaps the epilogue of tile t.
//
// Work: one CTA per work item, ordered heaviest first so the block scheduler
// balances the triangular work.  Row-LSE items are (query head, query tile),
// longest rows first.  Mass items are (KV head, key tile, query chunk of TPC
// tiles): a key row is split along the query axis into chunks whose partial
// sums go to the workspace and are added in fixed order by a reduce kernel
// (deterministic).
#include <cuda.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <mutex>

#include "kvp_common.cuh"
#include "kvp_launch.h"
#include "tc_ptx.cuh"

namespace kvp {
namespace {

constexpr int BM = 128;            // rows of the fixed A tile (TMEM lanes)
constexpr int BN = 128;            // rows of a streamed B tile (TMEM columns per accumulator)
constexpr int NSTAGE = 2;          // B tiles in flight
constexpr int NACC = 2;            // TMEM accumulators

// Epilogue layout: warp w reads TMEM lanes 32*(w%4).. and column group w/4 of each tile (NCG
// groups of CW columns).  Two groups (8 warps) measured faster than four (16 warps of 32 columns,
// where the per-tile overhead doubles) for every pass.
template <int MODE>
struct Epi {
  static constexpr int NCG = 2;
  static constexpr int WARPS = 4 * NCG;
  static constexpr int CW = BN / NCG;
  static constexpr int PRODUCER = WARPS;
  static constexpr int MMA = WARPS + 1;
  static constexpr int THREADS = 32 * (WARPS + 2);
};
constexpr int TMEM_COLS = NACC * BN;             // 256

constexpr int EXT_K = 16;                        // extra MMA K-step of the mass pass
constexpr int EXT_BYTES = 128 * EXT_K * 2;       // one [128 x 16] 16-bit operand (4 KB)

// Shared-memory layout for head dim HD (the MMA K): a 128-row tile is HD/64 TMA boxes of
// 128 rows x 128 bytes (16 KB each, 128-byte swizzle).
template <int HD>
struct Smem {
  static_assert(HD == 64 || HD == 128, "head_dim 64 or 128");
  static constexpr int HALVES = HD / 64;
  static constexpr int HALF_BYTES = 128 * 64 * 2;
  static constexpr int TILE_BYTES = HALVES * HALF_BYTES;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + TILE_BYTES;
  static constexpr int OFF_BAR = OFF_B + NSTAGE * TILE_BYTES;
  static constexpr int OFF_MISC = OFF_BAR + 256;
  static constexpr int OFF_AEXT = OFF_MISC + 256;          // key-side extension: [1, 1, 1, 0, ...]
  static constexpr int OFF_BEXT = OFF_AEXT + EXT_BYTES;    // query-side extension per stage
  static constexpr int OFF_RED = OFF_BEXT + NSTAGE * EXT_BYTES;
  // Sparse LSE (the mass pass's extension area is free there): the two operands of the masking
  // K-step, [128 x 8] 16-bit rows of 16 bytes (A: one per query row; B: one per key of a stage),
  // a zero block the descriptors read as k = 8..15, then the ring of per-tile column data.
  static constexpr int SX_BYTES = 128 * 16;
  static constexpr int OFF_SXA = OFF_AEXT;
  static constexpr int OFF_SXB = OFF_SXA + SX_BYTES;                 // [NSTAGE]
  static constexpr int OFF_SXZ = OFF_SXB + NSTAGE * SX_BYTES;
  static constexpr int OFF_RANK = OFF_SXZ + SX_BYTES;
  // row-state exchange of the epilogue (NCG - 1 groups of [m | l] per row) + alignment slack
  static constexpr int BYTES = OFF_RED + (Epi<0>::NCG - 1) * 2 * BM * 4 + 1024;
};
// Sparse LSE pass: ranks of the last NRK key tiles (the extension operands are unused there).
constexpr int NRK = 8;
static_assert(Smem<128>::OFF_RANK + NRK * BN * 4 <= Smem<128>::OFF_RED &&
                  Smem<64>::OFF_RANK + NRK * BN * 4 <= Smem<64>::OFF_RED,
              "masking operands and rank ring must fit in the extension area");

// Byte offset of element (r, k) of a [128 x 16] K-major operand in 8 x 16-byte core matrices
// (core (r/8, k/8) at (r/8)*256 + (k/8)*128): the layout desc_noswz(addr, 128, 256) reads.
__device__ __forceinline__ int ext_off(int r, int k) {
  return (r >> 3) * 256 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2;
}

// Round to bf16 / f16 (bits) and return the value kept.
__device__ __forceinline__ uint16_t round16(float x, bool bf16, float& kept) {
  if (bf16) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    kept = __bfloat162float(h);
    return *reinterpret_cast<const uint16_t*>(&h);
  }
  const __half h = __float2half_rn(x);
  kept = __half2float(h);
  return *reinterpret_cast<const uint16_t*>(&h);
}

struct TcParams {
  int S, Hq, Hkv, G;
  float c2;              // sm_scale * log2(e)
  float inv_scale;       // 1 / sm_scale
  int window;
  const float* lse;      // mass pass: natural-log row LSE [B*Hq*S]
  float* out;            // LSE pass: lse [B*Hq*S]; mass pass: partial sums (workspace)
  int n_groups;          // LSE pass: B*Hq; mass pass: B*Hkv
  int gblk;              // groups per block of the item order (decode_item)
  int NQT;               // LSE pass: query tiles per head
  int NT0, TPC, CMAX, NKT, Nf;   // mass pass schedule
  int per_head;          // mass pass: keep each query head's sum (partials [.., G, 2 halves, 128])
  // sparse LSE pass (MODE 2): static ranks and running cutoffs [B*Hkv*S] of the running top-k
  // mask; key j is kept for query i if j < n_sink, j > i - window, tau_i < 0 or rank_j <= tau_i
  const int32_t* ranks;
  const int32_t* tau;
  int n_sink;
  int ranks_vec;         // ranks rows are 16-byte aligned (S % 4 == 0): int4 loads
  // Rank-ordered stream of the sparse pass (null: dense streaming only): inv[B*Hkv*S] holds the
  // position of each rank (the inverse permutation) and the third tensor map the keys in rank
  // order; *perm_ok is zero when the ranks were not a permutation (then every tile is dense).
  const int32_t* inv;
  const int* perm_ok;
  // Rank-ordered tiles hold every key of rank <= the tile's largest cutoff, but only those at
  // positions the position-ordered tiles do not cover count there.  The others are masked in the
  // contraction: one more K = 16 step adds pen_a * pen_b (16-bit patterns of +2^a and -2^b,
  // c2 * 2^(a+b) >= 2^20) to their logits, so exp2 of them is exactly 0 and the epilogue tests
  // only the row's cutoff.  pen_a = 0: no masking step; the epilogue tests every key's position.
  uint32_t pen_a, pen_b;
  // a query tile takes the rank-ordered stream when it streams fewer than rank_bias_pct percent
  // of the dense causal row's tiles
  int rank_bias_pct;
  int* status;
  // persistent dense passes: the work-item counter (zero at launch) and the number of items
  int* queue;
  int total_items;
};

struct Item {
  int group;             // LSE: b*Hq+hq; mass: b*Hkv+h
  int tile;              // LSE: query tile qt; mass: key tile jt
  int chunk;             // mass: chunk index within the key row
  int per_head;          // mass: query tiles per head in this item
  int n_tiles;           // B tiles streamed by this CTA
};

// Work items are handed out in blocks of `gblk` groups: within a block the items of its groups
// are interleaved, heaviest first; blocks follow each other.  So the CTAs resident at one time
// work on a few groups whose streamed operand tiles (K for the LSE passes, Q for the mass
// pass) overlap and stay in L2, however many layers one launch covers.
template <int MODE>
__device__ __forceinline__ Item decode_item(int I, const TcParams& p) {
  Item it;
  if (MODE == 2) {
    // the sparse pass: plain heaviest-first order over every group (fewer live registers in a
    // kernel that is short of them)
    it.group = I % p.n_groups;
    it.tile = p.NQT - 1 - I / p.n_groups;
    it.chunk = 0;
    it.per_head = 0;
    it.n_tiles = it.tile + 1;
  } else if (MODE == 0) {
    const int per_block = p.NQT * p.gblk;
    const int blk = I / per_block, rem = I - blk * per_block;
    const int gb = min(p.gblk, p.n_groups - blk * p.gblk);
    it.group = blk * p.gblk + rem % gb;
    it.tile = p.NQT - 1 - rem / gb;
    it.chunk = 0;
    it.per_head = 0;
    it.n_tiles = it.tile + 1;
  } else {
    const long long full_total = (long long)p.Nf * p.n_groups;
    if (I < full_total) {
      const long long per_block = (long long)p.Nf * p.gblk;
      const int blk = (int)(I / per_block);
      const int rem = (int)(I - blk * per_block);
      const int gb = min(p.gblk, p.n_groups - blk * p.gblk);
      int local = rem / gb;
      it.group = blk * p.gblk + rem % gb;
      int c = 0;
      while (true) {
        const int n_c = p.NT0 - p.TPC * (c + 1) + 1;
        if (local < n_c) break;
        local -= n_c;
        ++c;
      }
      it.tile = local;
      it.chunk = c;
      it.per_head = p.TPC;
    } else {
      int local = (int)((I - full_total) / p.n_groups);
      it.group = (int)((I - full_total) % p.n_groups);
      it.tile = 0;
      it.chunk = 0;
      it.per_head = 0;
      for (int r = p.TPC - 1; r >= 1; --r) {
        const int cnt = p.NT0 >= r ? (p.NT0 - r) / p.TPC + 1 : 0;
        if (local < cnt) {
          it.tile = p.NT0 - r - local * p.TPC;
          it.chunk = local;
          it.per_head = r;
          break;
        }
        local -= cnt;
      }
    }
    it.n_tiles = it.per_head * p.G;
  }
  return it;
}

// Packed fp32 pairs (sm_100 family): two lanes of arithmetic per instruction.
__device__ __forceinline__ uint64_t pack2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <int MODE, int HD>
__global__ void __launch_bounds__(Epi<MODE>::THREADS, 2)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmE, const TcParams p, const bool bf16) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = ptx::smem_u32(smem);
  using L = Smem<HD>;
  constexpr int TILE_BYTES = L::TILE_BYTES, HALF_BYTES = L::HALF_BYTES;
  const uint32_t sA = s_base + L::OFF_A;
  const uint32_t sB = s_base + L::OFF_B;
  const uint32_t bar_full = s_base + L::OFF_BAR;                  // [NSTAGE]
  const uint32_t bar_empty = bar_full + 8 * NSTAGE;            // [NSTAGE]
  const uint32_t bar_accf = bar_empty + 8 * NSTAGE;            // [NACC]
  const uint32_t bar_acce = bar_accf + 8 * NACC;               // [NACC]
  const uint32_t bar_a = bar_acce + 8 * NACC;
  const uint32_t bar_rk = bar_a + 8;                           // [NRK] sparse LSE: ranks staged
  int* rbuf = reinterpret_cast<int*>(smem + L::OFF_RANK);         // [NRK][BN]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  float* red = reinterpret_cast<float*>(smem + L::OFF_RED);
  constexpr int EPI_WARPS = Epi<MODE>::WARPS, PRODUCER_WARP = Epi<MODE>::PRODUCER, MMA_WARP = Epi<MODE>::MMA;
  constexpr int NCG = Epi<MODE>::NCG, CW = Epi<MODE>::CW;
  const uint32_t sAext = s_base + L::OFF_AEXT;
  const uint32_t sBext = s_base + L::OFF_BEXT;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Item it = decode_item<MODE>(blockIdx.x, p);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      ptx::mbar_init(bar_full + 8 * s, 1);
      ptx::mbar_init(bar_empty + 8 * s, 1);
    }
    for (int a = 0; a < NACC; ++a) {
      ptx::mbar_init(bar_accf + 8 * a, 1);
      ptx::mbar_init(bar_acce + 8 * a, EPI_WARPS);
    }
    ptx::mbar_init(bar_a, 1);
    if (MODE == 2)
      for (int b = 0; b < NRK; ++b) ptx::mbar_init(bar_rk + 8 * b, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_holder), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  if (warp == PRODUCER_WARP && lane == 0) {
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmK);
  }
  if (MODE == 2 && p.pen_a != 0 && threadIdx.x < EPI_WARPS * 32) {
    // masking operand, query side: every row [2^a, 0 x 7]; and the zero block (k = 8..15)
    for (int e = threadIdx.x; e < 128; e += EPI_WARPS * 32) {
      *reinterpret_cast<uint4*>(smem + L::OFF_SXA + 16 * e) = make_uint4(p.pen_a, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(smem + L::OFF_SXZ + 16 * e) = make_uint4(0u, 0u, 0u, 0u);
    }
    ptx::fence_proxy_async_smem();
  }
  wait_prior_grid();                     // (sparse pass) the rank-ordered keys come from the kernel before
  int* tau_red = reinterpret_cast<int*>(smem + L::OFF_MISC + 16);      // sparse pass: [4] max, [4] min
  if (MODE == 2 && p.inv != nullptr && warp < 4) {
    // cutoff range over the query tile's rows (rows past S ignored)
    const int kvz = (it.group / p.Hq) * p.Hkv + (it.group % p.Hq) / p.G;
    const int i = it.tile * BM + threadIdx.x;
    const int tv = i < p.S ? __ldg(p.tau + (size_t)kvz * p.S + i) : -1;
    const int vmax = __reduce_max_sync(0xffffffffu, i < p.S ? tv : INT_MIN);
    const int vmin = __reduce_min_sync(0xffffffffu, i < p.S ? tv : INT_MAX);
    if (lane == 0) {
      tau_red[warp] = vmax;
      tau_red[4 + warp] = vmin;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  // Coordinates of the fixed A tile and of streamed tile t.  Q and K tensor maps are 4-D
  // (feature, token, head, batch); the A tile is (a_row, a_h, b_of_group).
  const int a_row = it.tile * BM;
  const int b_of_group = it.group / p.Hq;
  const int a_h = it.group % p.Hq;            // query head
  const int hkv = a_h / p.G;
  const int kv_z = b_of_group * p.Hkv + hkv;
  // Sparse pass, rank-ordered plan of a query tile whose rows all have a cutoff: the key tiles
  // holding the sinks and the protected windows in position order (eligible keys there are
  // dropped), then the keys in rank order up to the largest cutoff of the tile (eligible keys of
  // rank <= the row's cutoff are kept).  Used when it streams fewer tiles than the dense causal
  // row.
  bool rank_mode = false;
  int st_end = 0, wt0 = 0, n_pos = 0;
  const bool pen = MODE == 2 && p.pen_a != 0;
  if (MODE == 2 && p.inv != nullptr && *p.perm_ok) {
    const int i0 = it.tile * BM;
    const int tmax = max(max(tau_red[0], tau_red[1]), max(tau_red[2], tau_red[3]));
    const int tmin = min(min(tau_red[4], tau_red[5]), min(tau_red[6], tau_red[7]));
    if (tmin >= 0) {       // every row of the tile has a cutoff (the cutoffs need not be monotone)
      const int wlo = i0 - p.window + 1;
      wt0 = wlo > 0 ? wlo / BN : 0;
      const int sink_tiles = (p.n_sink + BN - 1) / BN;
      st_end = sink_tiles < wt0 ? sink_tiles : wt0;
      n_pos = st_end + (it.tile - wt0 + 1);
      const int n_rank = tmax / BN + 1;
      if ((n_pos + n_rank) * 100 < (it.tile + 1) * p.rank_bias_pct) {
        rank_mode = true;
        it.n_tiles = n_pos + n_rank;
      }
    }
  }
  // key tile (position order) of streamed tile t, or -1 for a rank-ordered tile
  auto key_tile = [&](int t) -> int {
    if (!rank_mode) return t;
    if (t < st_end) return t;
    if (t < n_pos) return wt0 + (t - st_end);
    return -1;
  };
  // token row of streamed key tile t in its tensor map (head hkv, batch b_of_group)
  auto b_row = [&](int t) -> int {
    const int kt = key_tile(t);
    return kt >= 0 ? kt * BN : (t - n_pos) * BN;
  };

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      ptx::mbar_arrive_expect_tx(bar_a, TILE_BYTES);
#pragma unroll
      for (int hb = 0; hb < L::HALVES; ++hb)
        ptx::tma_load_4d(sA + hb * HALF_BYTES, &tmQ, bar_a, 64 * hb, a_row, a_h, b_of_group);
    }
    if (MODE == 2 && lane == 0) ptx::prefetch_tmap(&tmE);
    int t = 0;
    for (; t < it.n_tiles; ++t) {
      const int s = t % NSTAGE, use = t / NSTAGE;
      bool ok = true;
      if (use > 0) ok = ptx::mbar_wait(bar_empty + 8 * s, (use - 1) & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (lane == 0) {
        const int row = b_row(t);
        const uint32_t dst = sB + s * TILE_BYTES;
        ptx::mbar_arrive_expect_tx(bar_full + 8 * s, TILE_BYTES);
        // sparse pass, rank-ordered tiles: the keys in rank order (third tensor map)
        const CUtensorMap* src = (MODE == 2 && rank_mode && key_tile(t) < 0) ? &tmE : &tmK;
#pragma unroll
        for (int hb = 0; hb < L::HALVES; ++hb)
          ptx::tma_load_4d(dst + hb * HALF_BYTES, src, bar_full + 8 * s, 64 * hb, row, hkv, b_of_group);
      }
      if (MODE == 2) {
        // Per-column data of the tile: the ranks of a position-ordered tile for the epilogue's
        // mask; of a rank-ordered tile, the masking step's B operand from the keys' positions.
        // (Without the masking step: +inf ranks for the sink and window tiles of the rank-ordered
        // plan and the positions of a rank-ordered tile, both for the epilogue.)
        const int kt = key_tile(t);
        if (rank_mode && kt < 0 && pen) {
          // rank-ordered tile: a key outside [st_end, wt0) tiles is counted by a position-ordered
          // tile (or lies past S): masked in the contraction through the B side of the masking
          // step of this stage
          const int kb = (t - n_pos) * BN + 4 * lane;
          const int32_t* src = p.inv + (size_t)kv_z * p.S + kb;
          int4 r4;
          if (p.ranks_vec && kb + 3 < p.S) {
            r4 = __ldg(reinterpret_cast<const int4*>(src));
          } else {
            r4.x = kb < p.S ? __ldg(src) : INT_MAX;
            r4.y = kb + 1 < p.S ? __ldg(src + 1) : INT_MAX;
            r4.z = kb + 2 < p.S ? __ldg(src + 2) : INT_MAX;
            r4.w = kb + 3 < p.S ? __ldg(src + 3) : INT_MAX;
          }
          const int lo = st_end * BN, hi = wt0 * BN;
          const uint32_t b0 = (r4.x < lo || r4.x >= hi) ? p.pen_b : 0u;
          const uint32_t b1 = (r4.y < lo || r4.y >= hi) ? p.pen_b : 0u;
          const uint32_t b2 = (r4.z < lo || r4.z >= hi) ? p.pen_b : 0u;
          const uint32_t b3 = (r4.w < lo || r4.w >= hi) ? p.pen_b : 0u;
          uint8_t* xb = smem + L::OFF_SXB + s * L::SX_BYTES + 16 * (4 * lane);
          *reinterpret_cast<uint4*>(xb) = make_uint4(b0, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(xb + 16) = make_uint4(b1, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(xb + 32) = make_uint4(b2, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(xb + 48) = make_uint4(b3, 0u, 0u, 0u);
          ptx::fence_proxy_async_smem();
        } else if (rank_mode && kt >= 0 && !pen) {
          *reinterpret_cast<int4*>(rbuf + (t % NRK) * BN + 4 * lane) = make_int4(INT_MAX, INT_MAX, INT_MAX, INT_MAX);
        } else {
          const int kb = (kt >= 0 ? kt : t - n_pos) * BN + 4 * lane;
          const int32_t* src = (rank_mode && kt < 0 ? p.inv : p.ranks) + (size_t)kv_z * p.S + kb;
          int4 r4;
          if (p.ranks_vec && kb + 3 < p.S) {
            r4 = __ldg(reinterpret_cast<const int4*>(src));
          } else {
            r4.x = kb < p.S ? __ldg(src) : INT_MAX;
            r4.y = kb + 1 < p.S ? __ldg(src + 1) : INT_MAX;
            r4.z = kb + 2 < p.S ? __ldg(src + 2) : INT_MAX;
            r4.w = kb + 3 < p.S ? __ldg(src + 3) : INT_MAX;
          }
          *reinterpret_cast<int4*>(rbuf + (t % NRK) * BN + 4 * lane) = r4;
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_rk + 8 * (t % NRK));
      }
    }
    if (lane == 0) {
      // Let every copy this warp started land before the CTA can exit.
      ptx::mbar_wait(bar_a, 0, abort_flag, p.status);
      for (int q = max(0, t - NSTAGE); q < t; ++q)
        ptx::mbar_wait(bar_full + 8 * (q % NSTAGE), (q / NSTAGE) & 1, abort_flag, p.status);
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_f16(bf16, BM, BN);
      int t = 0;
      if (ptx::mbar_wait(bar_a, 0, abort_flag, p.status)) {
        for (; t < it.n_tiles; ++t) {
          const int s = t % NSTAGE, a = t % NACC;
          if (!ptx::mbar_wait(bar_full + 8 * s, (t / NSTAGE) & 1, abort_flag, p.status)) break;
          if (t >= NACC && !ptx::mbar_wait(bar_acce + 8 * a, ((t / NACC) - 1) & 1, abort_flag, p.status))
            break;
          // rank-ordered tile with the masking step: its B operand is written by the producer
          const bool xt = pen && rank_mode && key_tile(t) < 0;
          if (xt && !ptx::mbar_wait(bar_rk + 8 * (t % NRK), (t / NRK) & 1, abort_flag, p.status)) break;
          ptx::tc_fence_after();
          const uint32_t d = tmem + a * BN;
          const uint32_t bs = sB + s * TILE_BYTES;
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * HALF_BYTES + (kk & 3) * 32;
            ptx::mma_f16_ss(d, ptx::desc_sw128(sA + off), ptx::desc_sw128(bs + off), idesc, kk > 0);
          }
          if (xt) {
            // rows of 16 bytes (core matrices 128 bytes apart); k = 8..15 read from the zero block
            const uint32_t xa = s_base + L::OFF_SXA, xb = s_base + L::OFF_SXB + s * L::SX_BYTES;
            const uint32_t xz = s_base + L::OFF_SXZ;
            ptx::mma_f16_ss(d, ptx::desc_noswz(xa, xz - xa, 128), ptx::desc_noswz(xb, xz - xb, 128), idesc, 1);
          }
          ptx::mma_commit(bar_empty + 8 * s);
          ptx::mma_commit(bar_accf + 8 * a);
        }
      }
      // The MMAs of the last issued tile must finish before TMEM is released.
      if (t > 0) ptx::mbar_wait(bar_accf + 8 * ((t - 1) % NACC), ((t - 1) / NACC) & 1, abort_flag, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int half = warp >> 2, quad = warp & 3;   // column group, TMEM lane quarter
    const int r = quad * 32 + lane;            // row of the A tile handled by this thread
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    float m = -INFINITY, l = 0.f;                            // running state (base 2)
    const int row_i = it.tile * BM + r;                       // LSE passes: query of this row
    int tau_eff = INT_MAX;                                   // sparse LSE: cutoff (none: INT_MAX)
    if (MODE == 2) {
      const int tq = row_i < p.S ? __ldg(p.tau + (size_t)kv_z * p.S + row_i) : -1;
      tau_eff = tq < 0 ? INT_MAX : tq;
    }
    bool ok = true;
    const uint64_t c2x2 = pack2(p.c2, p.c2);
    for (int t = 0; t < it.n_tiles; ++t) {
      const int a = t % NACC;
      if (!ptx::mbar_wait(bar_accf + 8 * a, (t / NACC) & 1, abort_flag, p.status)) { ok = false; break; }
      ptx::tc_fence_after();
      uint32_t v[CW];
      {
        const uint32_t taddr = tmem + lane_base + a * BN + half * CW;
#pragma unroll
        for (int h = 0; h < CW / 32; ++h)
          ptx::tmem_ld32(taddr + 32 * h, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * h]));
        ptx::tmem_ld_wait();
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_acce + 8 * a);

      {
        const int kt = key_tile(t);
        const bool diag = (kt == it.tile);
        if (diag) {
#pragma unroll
          for (int c = 0; c < CW; ++c)
            if (half * CW + c > r) v[c] = __float_as_uint(-INFINITY);
        }
        if (MODE == 2 && rank_mode && kt < 0 && pen) {
          // rank-ordered tile, keys outside the stream's position range already masked in the
          // contraction: column c (rank rb + c) is kept when its rank is within the row's cutoff
          const int cmax = tau_eff - ((t - n_pos) * BN + half * CW);
          if (cmax < 0) continue;
          if (cmax < CW - 1) {
#pragma unroll
            for (int c = 0; c < CW; ++c)
              if (c > cmax) v[c] = 0xff800000u;
          }
        } else if (MODE == 2 && rank_mode && kt < 0) {
          // rank-ordered tile: column c holds the key of rank rb + c at position pos[c]; kept
          // when that key is eligible for the row and its rank is within the row's cutoff
          if (!ptx::mbar_wait(bar_rk + 8 * (t % NRK), (t / NRK) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const int* ps = rbuf + (t % NRK) * BN + half * CW;
          const int cmax = tau_eff - ((t - n_pos) * BN + half * CW);   // rank within the cutoff: c <= cmax
          const int span = row_i - p.window - p.n_sink;                // eligible: 0 <= pos - n_sink <= span
#pragma unroll
          for (int g4 = 0; g4 < CW / 4; ++g4) {
            const int4 p4 = *reinterpret_cast<const int4*>(ps + 4 * g4);
            const int c = 4 * g4;
            const int d0 = p4.x - p.n_sink, d1 = p4.y - p.n_sink, d2 = p4.z - p.n_sink, d3 = p4.w - p.n_sink;
            if (d0 < 0 || d0 > span || c > cmax) v[c] = 0xff800000u;
            if (d1 < 0 || d1 > span || c + 1 > cmax) v[c + 1] = 0xff800000u;
            if (d2 < 0 || d2 > span || c + 2 > cmax) v[c + 2] = 0xff800000u;
            if (d3 < 0 || d3 > span || c + 3 > cmax) v[c + 3] = 0xff800000u;
          }
        } else if (MODE == 2) {
          // Columns cs <= c <= cw are eligible (neither sink nor in the protected window) and
          // are dropped when their rank is past the row's cutoff.  (Without the masking step the
          // sink and window tiles of the rank-ordered plan carry rank +inf: their eligible keys
          // are counted by the rank-ordered tiles.)
          const int jb = kt * BN + half * CW;
          const int cw = row_i - p.window - jb, cs = p.n_sink - jb;
          const int lo = cs > 0 ? cs : 0, hi = cw < CW - 1 ? cw : CW - 1;
          if (__any_sync(0xffffffffu, tau_eff != INT_MAX && lo <= hi)) {
            if (!ptx::mbar_wait(bar_rk + 8 * (t % NRK), (t / NRK) & 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            const int* rk = rbuf + (t % NRK) * BN + half * CW;
            if (__all_sync(0xffffffffu, lo == 0 && hi == CW - 1)) {
              // every column eligible for every row of the warp: the rank test alone
#pragma unroll
              for (int g4 = 0; g4 < CW / 4; ++g4) {
                const int4 r4 = *reinterpret_cast<const int4*>(rk + 4 * g4);
                v[4 * g4 + 0] = r4.x > tau_eff ? 0xff800000u : v[4 * g4 + 0];
                v[4 * g4 + 1] = r4.y > tau_eff ? 0xff800000u : v[4 * g4 + 1];
                v[4 * g4 + 2] = r4.z > tau_eff ? 0xff800000u : v[4 * g4 + 2];
                v[4 * g4 + 3] = r4.w > tau_eff ? 0xff800000u : v[4 * g4 + 3];
              }
            } else {
#pragma unroll
              for (int g4 = 0; g4 < CW / 4; ++g4) {
                const int4 r4 = *reinterpret_cast<const int4*>(rk + 4 * g4);
                const int rr[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const int c = 4 * g4 + u;
                  if (c >= lo && c <= hi && rr[u] > tau_eff) v[c] = 0xff800000u;
                }
              }
            }
          }
        }
        // sum over the tile of exp2(c2 * s - mref), four independent packed chains
        auto tile_sum = [&](float mref) -> float {
          const uint64_t nm2 = pack2(-mref, -mref);
          uint64_t s0 = 0, s1 = 0, s2 = 0, s3 = 0;
#pragma unroll
          for (int c = 0; c < CW; c += 8) {
            float x0, x1, x2, x3, x4, x5, x6, x7;
            unpack2(ffma2(pack2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])), c2x2, nm2), x0, x1);
            unpack2(ffma2(pack2(__uint_as_float(v[c + 2]), __uint_as_float(v[c + 3])), c2x2, nm2), x2, x3);
            unpack2(ffma2(pack2(__uint_as_float(v[c + 4]), __uint_as_float(v[c + 5])), c2x2, nm2), x4, x5);
            unpack2(ffma2(pack2(__uint_as_float(v[c + 6]), __uint_as_float(v[c + 7])), c2x2, nm2), x6, x7);
            s0 = fadd2(s0, pack2(fast_exp2(x0), fast_exp2(x1)));
            s1 = fadd2(s1, pack2(fast_exp2(x2), fast_exp2(x3)));
            s2 = fadd2(s2, pack2(fast_exp2(x4), fast_exp2(x5)));
            s3 = fadd2(s3, pack2(fast_exp2(x6), fast_exp2(x7)));
          }
          float q0, q1, q2, q3;
          unpack2(fadd2(s0, s1), q0, q1);
          unpack2(fadd2(s2, s3), q2, q3);
          return (q0 + q1) + (q2 + q3);
        };
        // Online normaliser against a lazily moved reference m (base 2): once a row has a kept
        // key the tile is summed against the current m without taking its max; only a sum that
        // reaches 2^64 (a term near overflow) sends the tile through the exact path (tile max,
        // rescale of l, sum), and l is brought back below 2^32 by exact power-of-two steps of m.
        // Terms that underflow against m are below 2^-126 of l >= 1.  In the sparse pass a score
        // masked by the masking step (about -2^20 after scaling) adds exactly 0 against any m a
        // kept key has set.
        bool exact = m == -INFINITY;
        if (!exact) {
          const float ts = tile_sum(m);
          if (ts < 0x1p64f) {
            l += ts;
            if (l >= 0x1p32f) {
              const int e = (int)((__float_as_uint(l) >> 23) & 0xffu) - 127;
              l *= __uint_as_float((uint32_t)(127 - e) << 23);
              m += (float)e;
            }
          } else {
            exact = true;
          }
        }
        if (exact) {
          float t0 = -INFINITY, t1 = -INFINITY, t2 = -INFINITY, t3 = -INFINITY;
#pragma unroll
          for (int c = 0; c < CW; c += 8) {
            t0 = max3(t0, __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
            t1 = max3(t1, __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
            t2 = max3(t2, __uint_as_float(v[c + 4]), __uint_as_float(v[c + 5]));
            t3 = max3(t3, __uint_as_float(v[c + 6]), __uint_as_float(v[c + 7]));
          }
          const float mn = fmaxf(m, fmaxf(fmaxf(t0, t1), fmaxf(t2, t3)) * p.c2);
          // (a tile whose only finite scores carry the masking step's -2^20 counts as empty)
          if (!(mn > (pen ? -0x1p19f : -INFINITY))) continue;
          if (mn > m) {
            l *= fast_exp2(m - mn);
            m = mn;
          }
          l += tile_sum(m);
        }
      }
    }
    // Combine the two column halves of every row and write the result.
    asm volatile("bar.sync 1, %0;" ::"r"(EPI_WARPS * 32));
    {
      if (half > 0) {
        red[(half - 1) * 2 * BM + r] = m;
        red[(half - 1) * 2 * BM + BM + r] = l;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(EPI_WARPS * 32));
      if (half == 0 && ok && !*abort_flag) {
        float M = m;
#pragma unroll
        for (int g = 1; g < NCG; ++g) M = fmaxf(M, red[(g - 1) * 2 * BM + r]);
        float L = 0.f;
        if (M != -INFINITY) {
          L = m == -INFINITY ? 0.f : l * fast_exp2(m - M);
#pragma unroll
          for (int g = 1; g < NCG; ++g) {
            const float mg = red[(g - 1) * 2 * BM + r], lg = red[(g - 1) * 2 * BM + BM + r];
            if (mg != -INFINITY) L += lg * fast_exp2(mg - M);
          }
        }
        const int i = it.tile * BM + r;
        if (i < p.S) p.out[(size_t)it.group * p.S + i] = (M + __log2f(L)) * KVP_LN2;
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- persistent mass pass
// The future-mass pass as persistent CTAs (two per SM, every one resident) that take work items
// from a global counter in the heaviest-first order of decode_item, so no CTA is set up per item:
//  * warp 8 (producer): fetches items one ahead and publishes each through a 4-slot item ring,
//    loads the item's key tile (A) once its buffer is free and streams its query tiles (B, with
//    their -lse/scale extension box) through a 2-stage ring;
//  * warp 9 (MMA, one thread): 128x128 tcgen05 products (+ the extension K-step) into two TMEM
//    accumulators, tile T into accumulator T % 2;
//  * warps 0-7 (epilogue): warp w reads TMEM lanes 32*(w%4).. and column half w/4 of every tile;
//    each (row, half) keeps its own partial sum and writes it to the workspace, where the
//    reduce kernel adds the halves and chunks in fixed order.
// Measured against one CTA per work item: 2-3 % faster on the Qwen3-4B layer and at S = 131072
// (the row-LSE pass measured slower in this form and keeps one CTA per item).  One CTA per SM
// with two epilogue groups on alternate tiles and all four accumulators measured 30 % slower:
// a single MMA stream per SM does not keep the tensor pipe busy.
constexpr int P_EPI_WARPS = 8;
constexpr int P_PRODUCER = P_EPI_WARPS;
constexpr int P_MMA = P_EPI_WARPS + 1;
constexpr int P_THREADS = 32 * (P_EPI_WARPS + 2);
constexpr int P_CTAS_PER_SM = 2;
constexpr int P_NACC = 2;                      // TMEM accumulators
constexpr int P_NSTAGE = 2;                    // B tiles in flight
constexpr int P_NITEM = 4;                     // published work items
constexpr int P_TMEM_COLS = P_NACC * BN;       // 256
constexpr int P_SLOTS = 2;                     // partial sums per row of an item: one per column half

template <int HD>
struct PSmem {
  static constexpr int HALVES = HD / 64;
  static constexpr int HALF_BYTES = 128 * 64 * 2;
  static constexpr int TILE_BYTES = HALVES * HALF_BYTES;
  static constexpr int OFF_A = 0;                                    // key tile
  static constexpr int OFF_B = OFF_A + TILE_BYTES;                   // [P_NSTAGE] query tiles
  static constexpr int OFF_BEXT = OFF_B + P_NSTAGE * TILE_BYTES;     // [P_NSTAGE] query-side extension
  static constexpr int OFF_AEXT = OFF_BEXT + P_NSTAGE * EXT_BYTES;   // key-side extension
  static constexpr int OFF_BAR = OFF_AEXT + EXT_BYTES;
  static constexpr int OFF_MISC = OFF_BAR + 8 * (2 * P_NSTAGE + 2 * P_NACC + 2 + 2 * P_NITEM);
  static constexpr int BYTES = OFF_MISC + 64 + 1024;                 // + alignment slack
  static_assert(P_CTAS_PER_SM * (BYTES + 1024) <= 228 * 1024, "the CTAs of one SM must fit its shared memory");
};

template <int HD>
__global__ void __launch_bounds__(P_THREADS, P_CTAS_PER_SM)
    mass_tc_persistent_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                              const __grid_constant__ CUtensorMap tmE, const TcParams p, const bool bf16) {
  using L = PSmem<HD>;
  constexpr int TILE_BYTES = L::TILE_BYTES, HALF_BYTES = L::HALF_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = ptx::smem_u32(smem);
  const uint32_t sA = s_base + L::OFF_A, sB = s_base + L::OFF_B;
  const uint32_t sAext = s_base + L::OFF_AEXT, sBext = s_base + L::OFF_BEXT;
  const uint32_t bar_bfull = s_base + L::OFF_BAR;              // [P_NSTAGE]
  const uint32_t bar_bempty = bar_bfull + 8 * P_NSTAGE;        // [P_NSTAGE]
  const uint32_t bar_accf = bar_bempty + 8 * P_NSTAGE;         // [P_NACC]
  const uint32_t bar_acce = bar_accf + 8 * P_NACC;             // [P_NACC]
  const uint32_t bar_afull = bar_acce + 8 * P_NACC;
  const uint32_t bar_aempty = bar_afull + 8;
  const uint32_t bar_ifull = bar_aempty + 8;                   // [P_NITEM]
  const uint32_t bar_iempty = bar_ifull + 8 * P_NITEM;         // [P_NITEM]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  volatile int* ring = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 16);   // [P_NITEM]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_NSTAGE; ++s) {
      ptx::mbar_init(bar_bfull + 8 * s, 1);
      ptx::mbar_init(bar_bempty + 8 * s, 1);
    }
    for (int a = 0; a < P_NACC; ++a) {
      ptx::mbar_init(bar_accf + 8 * a, 1);
      ptx::mbar_init(bar_acce + 8 * a, P_EPI_WARPS);
    }
    ptx::mbar_init(bar_afull, 1);
    ptx::mbar_init(bar_aempty, 1);
    for (int q = 0; q < P_NITEM; ++q) {
      ptx::mbar_init(bar_ifull + 8 * q, 1);
      ptx::mbar_init(bar_iempty + 8 * q, 2);                     // the MMA thread and the epilogue
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == P_MMA) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_holder), P_TMEM_COLS);
    ptx::tmem_relinquish();
  }
  if (threadIdx.x < P_EPI_WARPS * 32) {
    // The extra K-step adds -lse_i/scale (B side, three 16-bit parts) times 1 (A side) to every
    // logit, so the accumulator holds the LSE-offset logit: the key-side extension
    // [1, 1, 1, 0, ...] is written once; of the query-side extension of every stage TMA writes
    // the lower half (k = 0..7) and the upper half stays zero.
    const uint16_t one = bf16 ? 0x3F80u : 0x3C00u;
    for (int e = threadIdx.x; e < 128 * EXT_K; e += P_EPI_WARPS * 32) {
      const int r = e / EXT_K, k = e % EXT_K;
      *reinterpret_cast<uint16_t*>(smem + L::OFF_AEXT + ext_off(r, k)) = k < 3 ? one : 0u;
    }
    for (int e = threadIdx.x; e < P_NSTAGE * EXT_BYTES / 16; e += P_EPI_WARPS * 32) {
      const int st = e / (EXT_BYTES / 16), off = (e % (EXT_BYTES / 16)) * 16;
      if (off >= EXT_BYTES / 2) *reinterpret_cast<uint4*>(smem + L::OFF_BEXT + st * EXT_BYTES + off) = make_uint4(0u, 0u, 0u, 0u);
    }
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  wait_prior_grid();                     // the extension rows and the queue come from ext_prep

  if (warp == P_PRODUCER) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmE);
      int next = atomicAdd(p.queue, 1);
      long long T = 0;
      int i = 0, last_a = -1;
      for (;; ++i) {
        const int slot = i % P_NITEM;
        if (i >= P_NITEM && !ptx::mbar_wait(bar_iempty + 8 * slot, ((i / P_NITEM) - 1) & 1, abort_flag, p.status))
          break;
        const int I = next < p.total_items ? next : -1;
        ring[slot] = I;
        ptx::mbar_arrive(bar_ifull + 8 * slot);                 // release: the entry is visible
        if (I < 0) break;
        next = atomicAdd(p.queue, 1);                           // the following item, ahead of time
        const Item it = decode_item<1>(I, p);
        const int b_of_group = it.group / p.Hkv, hkv = it.group % p.Hkv;
        if (i >= 1 && !ptx::mbar_wait(bar_aempty, (i - 1) & 1, abort_flag, p.status)) break;
        ptx::mbar_arrive_expect_tx(bar_afull, TILE_BYTES);
#pragma unroll
        for (int hb = 0; hb < L::HALVES; ++hb)
          ptx::tma_load_4d(sA + hb * HALF_BYTES, &tmK, bar_afull, 64 * hb, it.tile * BM, hkv, b_of_group);
        last_a = i;
        bool ok = true;
        int gh = 0, u = 0;
        for (int t = 0; t < it.n_tiles; ++t, ++T) {
          const int s = (int)(T % P_NSTAGE);
          if (T >= P_NSTAGE && !ptx::mbar_wait(bar_bempty + 8 * s, ((T / P_NSTAGE) - 1) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          // streamed tile t is query tile u of query head gh of the group
          const int row = it.tile * BM + p.window + BN * (it.chunk * p.TPC + u);
          const int h = hkv * p.G + gh;
          if (++u == it.per_head) {
            u = 0;
            ++gh;
          }
          const uint32_t dst = sB + s * TILE_BYTES;
          ptx::mbar_arrive_expect_tx(bar_bfull + 8 * s, TILE_BYTES + EXT_BYTES / 2);
#pragma unroll
          for (int hb = 0; hb < L::HALVES; ++hb)
            ptx::tma_load_4d(dst + hb * HALF_BYTES, &tmQ, bar_bfull + 8 * s, 64 * hb, row, h, b_of_group);
          ptx::tma_load_3d(sBext + s * EXT_BYTES, &tmE, bar_bfull + 8 * s, 0, row, b_of_group * p.Hq + h);
        }
        if (!ok) break;
      }
      // copies still in flight land before the CTA can exit
      if (last_a >= 0) ptx::mbar_wait_drain(bar_afull, last_a & 1, p.status);
      for (long long q = T - P_NSTAGE < 0 ? 0 : T - P_NSTAGE; q < T; ++q)
        ptx::mbar_wait_drain(bar_bfull + 8 * (int)(q % P_NSTAGE), (q / P_NSTAGE) & 1, p.status);
    }
  } else if (warp == P_MMA) {
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_f16(bf16, BM, BN);
      long long T = 0;
      for (int i = 0;; ++i) {
        const int slot = i % P_NITEM;
        if (!ptx::mbar_wait(bar_ifull + 8 * slot, (i / P_NITEM) & 1, abort_flag, p.status)) break;
        const int I = ring[slot];
        ptx::mbar_arrive(bar_iempty + 8 * slot);
        if (I < 0) break;
        const Item it = decode_item<1>(I, p);
        if (!ptx::mbar_wait(bar_afull, i & 1, abort_flag, p.status)) break;
        ptx::tc_fence_after();
        bool ok = true;
        for (int t = 0; t < it.n_tiles; ++t, ++T) {
          const int s = (int)(T % P_NSTAGE), a = (int)(T % P_NACC);
          if (!ptx::mbar_wait(bar_bfull + 8 * s, (T / P_NSTAGE) & 1, abort_flag, p.status) ||
              (T >= P_NACC && !ptx::mbar_wait(bar_acce + 8 * a, ((T / P_NACC) - 1) & 1, abort_flag, p.status))) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d = tmem + a * BN;
          const uint32_t bs = sB + s * TILE_BYTES;
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * HALF_BYTES + (kk & 3) * 32;
            ptx::mma_f16_ss(d, ptx::desc_sw128(sA + off), ptx::desc_sw128(bs + off), idesc, kk > 0);
          }
          ptx::mma_f16_ss(d, ptx::desc_noswz(sAext, 128, 256), ptx::desc_noswz(sBext + s * EXT_BYTES, 2048, 128),
                          idesc, 1);
          ptx::mma_commit(bar_bempty + 8 * s);
          ptx::mma_commit(bar_accf + 8 * a);
        }
        if (!ok) break;
        ptx::mma_commit(bar_aempty);                            // the key tile is free once these complete
      }
      // the last products must be complete before TMEM is released
      if (T > 0) ptx::mbar_wait_drain(bar_accf + 8 * (int)((T - 1) % P_NACC), ((T - 1) / P_NACC) & 1, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int half = warp >> 2, quad = warp & 3;
    constexpr int CW = BN / 2;
    const int r = quad * 32 + lane;                             // key row of the A tile
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint64_t c2x2 = pack2(p.c2, p.c2);
    long long T = 0;
    for (int i = 0;; ++i) {
      const int slot = i % P_NITEM;
      const bool got = ptx::mbar_wait(bar_ifull + 8 * slot, (i / P_NITEM) & 1, abort_flag, p.status);
      const int I = got ? ring[slot] : -1;
      // every warp reads the entry before one thread releases it; a failed wait ends the loop
      // of every epilogue warp together
      if (ptx::bar_red_or(I < 0, 1, P_EPI_WARPS * 32)) break;
      if (threadIdx.x == 0) ptx::mbar_arrive(bar_iempty + 8 * slot);
      const Item it = decode_item<1>(I, p);
      uint64_t acc01 = 0, acc23 = 0;                            // packed partial sums
      // per query head: the head the accumulator holds (-1: none), the next unwritten head
      int acc_head = -1, hd_next = 0;
      float* part = p.out + ((((size_t)it.group * p.NKT + it.tile) * p.CMAX + it.chunk) *
                             (p.per_head ? p.G : 1)) * P_SLOTS * BM;
      auto write_head = [&](int h) {
        float f0, f1, f2, f3;
        unpack2(acc01, f0, f1);
        unpack2(acc23, f2, f3);
        for (; hd_next < h; ++hd_next) part[((size_t)hd_next * P_SLOTS + half) * BM + r] = 0.f;
        part[((size_t)h * P_SLOTS + half) * BM + r] = (f0 + f1) + (f2 + f3);
        hd_next = h + 1;
        acc01 = 0;
        acc23 = 0;
      };
      bool ok = true;
      int gh = 0, u = 0;
      for (int t = 0; t < it.n_tiles; ++t) {
        const int tgh = gh, tu = u;
        if (++u == it.per_head) {
          u = 0;
          ++gh;
        }
        const long long TT = T + t;
        const int a = (int)(TT % P_NACC);
        if (!ptx::mbar_wait(bar_accf + 8 * a, (TT / P_NACC) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        uint32_t v[CW];
        {
          const uint32_t taddr = tmem + lane_base + a * BN + half * CW;
#pragma unroll
          for (int h = 0; h < CW / 32; ++h)
            ptx::tmem_ld32(taddr + 32 * h, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * h]));
          ptx::tmem_ld_wait();
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_acce + 8 * a);
        if (p.per_head) {                                       // a new head: the previous one is complete
          if (acc_head >= 0 && tgh != acc_head) write_head(acc_head);
          acc_head = tgh;
        }
        // the accumulator holds (q.k - lse_i/scale); past S it is -inf
        if (it.chunk == 0 && tu == 0) {                         // the window-diagonal tile: i >= j + w
#pragma unroll
          for (int c = 0; c < CW; ++c)
            if (half * CW + c < r) v[c] = __float_as_uint(-INFINITY);
        }
        const uint64_t zero2 = 0;
#pragma unroll
        for (int c = 0; c < CW; c += 4) {
          float x0, x1, x2, x3;
          unpack2(ffma2(pack2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])), c2x2, zero2), x0, x1);
          unpack2(ffma2(pack2(__uint_as_float(v[c + 2]), __uint_as_float(v[c + 3])), c2x2, zero2), x2, x3);
          acc01 = fadd2(acc01, pack2(fast_exp2(x0), fast_exp2(x1)));
          acc23 = fadd2(acc23, pack2(fast_exp2(x2), fast_exp2(x3)));
        }
      }
      if (ok) {
        if (p.per_head) {
          if (acc_head >= 0) write_head(acc_head);
          for (; hd_next < p.G; ++hd_next) part[((size_t)hd_next * P_SLOTS + half) * BM + r] = 0.f;
        } else {
          float f0, f1, f2, f3;
          unpack2(acc01, f0, f1);
          unpack2(acc23, f2, f3);
          part[(size_t)half * BM + r] = (f0 + f1) + (f2 + f3);
        }
      }
      if (ptx::bar_red_or(!ok || *abort_flag != 0, 1, P_EPI_WARPS * 32)) break;
      T += it.n_tiles;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == P_MMA) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, P_TMEM_COLS);
  }
}

// Query-side extension of the mass pass: row i of head z holds -lse[z, i]/scale split into three
// 16-bit parts (exactly representable sum to ~2^-24 relative), then zeros; rows i >= S (the
// padding the last query tiles read) hold -inf, so those queries get weight exactly 0.
__global__ void ext_prep_kernel(const float* __restrict__ lse, int BHq, int S, int S_pad,
                                float inv_scale, bool bf16, uint4* __restrict__ ext, int* queue) {
  wait_prior_grid();                     // lse may come from the kernel just before
  if (blockIdx.x == 0 && threadIdx.x == 0) *queue = 0;   // the mass pass's work counter
  const long long total = (long long)BHq * S_pad;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int z = (int)(e / S_pad), i = (int)(e % S_pad);
    uint16_t h1, h2 = 0, h3 = 0;
    if (i >= S) {
      h1 = bf16 ? 0xFF80u : 0xFC00u;
    } else {
      const float h = -lse[(size_t)z * S + i] * inv_scale;
      float k1, k2, k3;
      h1 = round16(h, bf16, k1);
      h2 = round16(h - k1, bf16, k2);
      h3 = round16((h - k1) - k2, bf16, k3);
    }
    ext[e] = make_uint4((uint32_t)h1 | ((uint32_t)h2 << 16), (uint32_t)h3, 0u, 0u);
  }
}

// Sparse pass, rank-ordered stream, in one scatter over the keys: inv[h, rank[h, j]] = j and
// ks[h, rank[h, j]] = k[h, j] (ks dense [B*Hkv, S, D]; k read through its element strides).
// inv starts at -1; a rank outside [0, S) or a rank met twice (the previous inv entry was already
// set) clears *ok.  S in-range ranks without a repeat are a permutation, so *ok stays nonzero
// exactly when ks and inv are complete.
__global__ void rank_scatter_keys_kernel(const uint16_t* __restrict__ k, long long k_sb, long long k_sh,
                                         long long k_sr, int Hkv, const int32_t* __restrict__ ranks,
                                         int S, int vpr, long long total, int32_t* __restrict__ inv,
                                         uint4* __restrict__ ks, int* ok) {
  wait_prior_grid();
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const long long hj = e / vpr;                    // h * S + j, h = b * Hkv + hk
    const int c = (int)(e - hj * vpr);
    const long long h = hj / S;
    const int j = (int)(hj - h * S);
    const int r = ranks[hj];
    if ((unsigned)r >= (unsigned)S) {
      if (c == 0) *ok = 0;
      continue;
    }
    if (c == 0 && atomicExch(inv + h * S + r, j) != -1) *ok = 0;
    const uint16_t* src = k + (h / Hkv) * k_sb + (h % Hkv) * k_sh + (long long)j * k_sr;
    ks[(h * S + r) * vpr + c] = reinterpret_cast<const uint4*>(src)[c];
  }
}

// F[group, j] = the partial sums of key tile j/128: its chunks in order, each chunk's two
// column-half slots in order (deterministic).
__global__ void __launch_bounds__(BM) fam_reduce_kernel(const float* __restrict__ part, int S, int NT0,
                                                        int TPC, int CMAX, int NKT,
                                                        float* __restrict__ F) {
  wait_prior_grid();
  const int jt = blockIdx.x, group = blockIdx.y, r = threadIdx.x;
  const int j = jt * BM + r;
  if (j >= S) return;
  const int nt = max(0, NT0 - jt);
  const int nch = (nt + TPC - 1) / TPC;
  const float* src = part + ((size_t)group * NKT + jt) * CMAX * P_SLOTS * BM + r;
  float f = 0.f;
  for (int c = 0; c < nch; ++c)
#pragma unroll
    for (int q = 0; q < P_SLOTS; ++q) f += src[((size_t)c * P_SLOTS + q) * BM];
  F[(size_t)group * S + j] = f;
}

// Per-head mode of the mass pass, reduce and KVpop target in one pass: each query head's sum
// over its chunks and slots in order (F_heads), then N_t = max(1, S - (j + w)) and the group max
// of log(eps + F_g / N_t) or log(eps + sum_g F_g / (N_t G)) (target), and the group sum (F);
// each written when given.  The arithmetic of the target is that of target_epilogue_kernel.
__global__ void __launch_bounds__(BM) fam_target_kernel(const float* __restrict__ part, int S, int Hkv, int G,
                                                        int NT0, int TPC, int CMAX, int NKT, int window,
                                                        float eps, int aggregate, float* __restrict__ F_heads,
                                                        float* __restrict__ target, float* __restrict__ F) {
  wait_prior_grid();
  const int jt = blockIdx.x, group = blockIdx.y, r = threadIdx.x;
  const int j = jt * BM + r;
  if (j >= S) return;
  const int nt = max(0, NT0 - jt);
  const int nch = (nt + TPC - 1) / TPC;
  const int b = group / Hkv, h = group % Hkv;
  const float N = (float)max(1, S - (j + window));
  float sum = 0.f, best = -INFINITY;
  for (int g = 0; g < G; ++g) {
    float f = 0.f;
    for (int c = 0; c < nch; ++c) {
      const float* src = part + ((((size_t)group * NKT + jt) * CMAX + c) * G + g) * P_SLOTS * BM + r;
#pragma unroll
      for (int q = 0; q < P_SLOTS; ++q) f += src[(size_t)q * BM];
    }
    if (F_heads) F_heads[((size_t)b * Hkv * G + h * G + g) * S + j] = f;
    sum += f;
    best = fmaxf(best, logf(eps + f / N));
  }
  const size_t e = (size_t)group * S + j;
  if (target) target[e] = aggregate == 0 ? best : logf(eps + sum / (N * (float)G));
  if (F) F[e] = sum;
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// [n_batch, n_heads, S, D] tensor with element strides (sb, sh, sr) (D contiguous) as a 4-D map
// (feature, token, head, batch): 128-row x 64-element boxes, 128-byte swizzle, zero fill past S.
// The stride of a dimension of extent 1 is never applied; it is replaced by a valid value.
bool make_tmap(CUtensorMap* m, const void* base, int dtype, int D, int S, int n_heads, int n_batch,
               long long sr, long long sh, long long sb) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  if (n_heads == 1) sh = sr * S;
  if (n_batch == 1) sb = sh * n_heads;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)n_heads, (cuuint64_t)n_batch};
  cuuint64_t strides[3] = {(cuuint64_t)sr * 2, (cuuint64_t)sh * 2, (cuuint64_t)sb * 2};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt =
      dtype == KVP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool make_q_tmap(CUtensorMap* m, const void* q, int dtype, const AttnShape& s) {
  return make_tmap(m, q, dtype, s.head_dim, s.seq_len, s.h_q, s.n_batch, s.q_sr, s.q_sh, s.q_sb);
}
bool make_k_tmap(CUtensorMap* m, const void* k, int dtype, const AttnShape& s) {
  return make_tmap(m, k, dtype, s.head_dim, s.seq_len, s.h_kv, s.n_batch, s.k_sr, s.k_sh, s.k_sb);
}

// Tensor map of the mass pass's query-side extension [n_heads, S_pad, 8] (16-byte rows, boxes of
// 128 rows, no swizzle: a box lands as 128 contiguous 16-byte rows).
bool make_ext_tmap(CUtensorMap* m, const void* base, int dtype, int n_heads, int S_pad) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {8, (cuuint64_t)S_pad, (cuuint64_t)n_heads};
  cuuint64_t strides[2] = {16, (cuuint64_t)S_pad * 16};
  cuuint32_t box[3] = {8, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt =
      dtype == KVP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct FamSched {
  int NT0, TPC, CMAX, NKT, Nf, Np;
};

FamSched fam_schedule(AttnShape s, int window) {
  FamSched f{};
  const int n_groups = s.n_batch * s.h_kv;
  f.NKT = (s.seq_len + BM - 1) / BM;
  f.NT0 = s.seq_len > window ? (s.seq_len - window + BN - 1) / BN : 0;
  // Chunk length (query tiles per head per item): enough items for ~8 per SM.
  const double tiles = 0.5 * (double)n_groups * f.NT0 * (f.NT0 + 1);
  int tpc = 64;
  while (tpc > 2 && tiles / tpc < 8.0 * 152) tpc >>= 1;
  f.TPC = tpc;
  f.CMAX = std::max(1, (f.NT0 + tpc - 1) / tpc);
  f.Nf = 0;
  for (int c = 0;; ++c) {
    const int n_c = f.NT0 - tpc * (c + 1) + 1;
    if (n_c <= 0) break;
    f.Nf += n_c;
  }
  f.Np = 0;
  for (int r = 1; r < tpc; ++r)
    if (f.NT0 >= r) f.Np += (f.NT0 - r) / tpc + 1;
  return f;
}

template <int MODE, int HD>
cudaError_t launch_tc_hd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& te, const TcParams& p,
                         int grid, bool bf16, cudaStream_t st) {
  auto kern = attn_tc_kernel<MODE, HD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<HD>::BYTES);
  if (e != cudaSuccess) return e;
  count_launches(1);
  if (MODE == 2 && p.inv != nullptr)       // after its preparation scatter: dependent launch
    return launch_with_pdl(kern, dim3(grid), dim3(Epi<MODE>::THREADS), Smem<HD>::BYTES, st, tq, tk, te, p, bf16);
  kern<<<grid, Epi<MODE>::THREADS, Smem<HD>::BYTES, st>>>(tq, tk, te, p, bf16);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_tc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& te, const TcParams& p,
                      int grid, bool bf16, int head_dim, cudaStream_t st) {
  return head_dim == 64 ? launch_tc_hd<MODE, 64>(tq, tk, te, p, grid, bf16, st)
                        : launch_tc_hd<MODE, 128>(tq, tk, te, p, grid, bf16, st);
}

template <int HD>
cudaError_t launch_mass_persistent_hd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& te,
                                      const TcParams& p, bool bf16, cudaStream_t st) {
  auto kern = mass_tc_persistent_kernel<HD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PSmem<HD>::BYTES);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int slots = P_CTAS_PER_SM * sms;                        // every CTA resident at once
  const int grid = p.total_items < slots ? p.total_items : slots;
  count_launches(1);
  return launch_with_pdl(kern, dim3(grid), dim3(P_THREADS), PSmem<HD>::BYTES, st, tq, tk, te, p, bf16);
}

}  // namespace

bool tc_encoder_available() { return encode_fn() != nullptr; }

size_t sparse_lse_workspace_size(int dtype, AttnShape s) {
  if (dtype != KVP_BF16 && dtype != KVP_F16) return 0;
  const size_t n = (size_t)s.n_batch * s.h_kv * s.seq_len;
  return ((n * 4 + 255) & ~(size_t)255) + ((n * s.head_dim * 2 + 255) & ~(size_t)255) + 256;
}

// Workspace of the mass pass: partial sums (P_SLOTS per row of every item chunk, per query head
// in the per-head mode), the query-side extension (16 bytes per query row, S + 128 rows per
// query head), then the work-item counter.
size_t fam_partial_bytes(AttnShape s, const FamSched& f, int per_head) {
  const size_t heads = per_head ? (size_t)(s.h_q / s.h_kv) : 1;
  return (((size_t)s.n_batch * s.h_kv * f.NKT * f.CMAX * heads * P_SLOTS * BM * sizeof(float)) + 255) &
         ~(size_t)255;
}

size_t fam_ext_bytes(AttnShape s) {
  return (((size_t)s.n_batch * s.h_q * (s.seq_len + BN) * 16) + 255) & ~(size_t)255;
}

size_t fam_tc_workspace_size(AttnShape s, int window, int per_head) {
  const FamSched f = fam_schedule(s, window);
  return fam_partial_bytes(s, f, per_head) + fam_ext_bytes(s) + 256;
}

// Bit patterns of +2^a and -2^b for the sparse pass's masking step: a + b = e, the smallest e
// with c2 * 2^e >= 2^20 (so a masked score's exp2 underflows to exactly 0 and the rounding of
// c2 * 2^e stays far below one unit of the exponent).  Both 0 when 2^a or 2^b is not a normal
// number of the operand type; the kernel then tests every key's position instead.
void masking_step_bits(float c2, bool bf16, uint32_t* pa, uint32_t* pb) {
  *pa = *pb = 0;
  if (!(c2 > 0.f) || !std::isfinite(c2)) return;
  const int e = (int)std::ceil(20.0 - std::log2((double)c2));
  const int a = (int)std::floor(e / 2.0), b = e - a;
  const int lo = bf16 ? -126 : -14, hi = bf16 ? 127 : 15;
  if (a < lo || a > hi || b < lo || b > hi) return;
  *pa = bf16 ? (uint32_t)(a + 127) << 7 : (uint32_t)(a + 15) << 10;
  *pb = (bf16 ? (uint32_t)(b + 127) << 7 : (uint32_t)(b + 15) << 10) | 0x8000u;
}

cudaError_t launch_lse_tc(const void* q, const void* k, int dtype, AttnShape s, float scale,
                          float* lse, int* status, cudaStream_t st, const SparseMask* mask) {
  CUtensorMap tq, tk;
  if (!make_q_tmap(&tq, q, dtype, s) || !make_k_tmap(&tk, k, dtype, s)) return cudaErrorInvalidValue;
  TcParams p{};
  p.S = s.seq_len;
  p.Hq = s.h_q;
  p.Hkv = s.h_kv;
  p.G = s.h_q / s.h_kv;
  p.c2 = scale * KVP_LOG2E;
  p.out = lse;
  p.n_groups = s.n_batch * s.h_q;
  // Items in blocks of up to 32 query heads whose keys together stay within about 96 MB of L2
  // (32 at S <= 32768; 8 at S = 131072, where the pass takes 47.5 instead of 48.6 ms).
  {
    const double k_head = (double)s.seq_len * s.head_dim * 2;
    const int gb = std::max(1, std::min(32, (int)(96e6 / k_head) * (s.h_q / s.h_kv)));
    p.gblk = std::min(p.n_groups, gb);
  }
  p.NQT = (s.seq_len + BM - 1) / BM;
  p.status = status;
  const bool bf16 = dtype == KVP_BF16;
  if (mask) {
    p.ranks = mask->ranks;
    p.tau = mask->tau;
    p.n_sink = mask->n_sink;
    p.window = mask->window;
    p.ranks_vec = s.seq_len % 4 == 0 && ((uintptr_t)mask->ranks & 15) == 0;
    if (!mask->inv) return launch_tc<2>(tq, tk, tk, p, p.n_groups * p.NQT, bf16, s.head_dim, st);
    // rank-ordered stream: inverse permutation, keys in rank order, validity flag
    const int BHkv = s.n_batch * s.h_kv;
    const long long n = (long long)BHkv * s.seq_len;
    cudaError_t e = cudaMemsetAsync(mask->inv, 0xFF, (size_t)n * sizeof(int32_t), st);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(mask->perm_ok, 1, sizeof(int), st);      // nonzero until a check fails
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int vpr = s.head_dim * 2 / 16;
    const long long cap = (long long)sms * 8;
    long long b2 = (n * vpr + 255) / 256;
    b2 = b2 > cap ? cap : b2;
    count_launches(1);
    rank_scatter_keys_kernel<<<(unsigned)b2, 256, 0, st>>>((const uint16_t*)k, s.k_sb, s.k_sh, s.k_sr, s.h_kv,
                                                           mask->ranks, s.seq_len, vpr, n * vpr, mask->inv,
                                                           (uint4*)mask->k_sorted, mask->perm_ok);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap tks;
    const long long sd = (long long)s.seq_len * s.head_dim;
    if (!make_tmap(&tks, mask->k_sorted, dtype, s.head_dim, s.seq_len, s.h_kv, s.n_batch, s.head_dim, sd,
                   sd * s.h_kv))
      return cudaErrorInvalidValue;
    p.inv = mask->inv;
    p.perm_ok = mask->perm_ok;
    masking_step_bits(p.c2, bf16, &p.pen_a, &p.pen_b);
    // With the masking step a rank-ordered tile costs less than a dense one with its per-score
    // rank test, so the rank-ordered stream pays even when it is somewhat longer (Qwen3-4B layer,
    // k = 1916 of 8192: 0.220 / 0.214 / 0.214 / 0.216 / 0.222 ms at 100 / 130 / 160 / 200 / 260 %).
    // Without it (pen_a = 0) a rank-ordered tile tests every key's position: shorter streams only.
    p.rank_bias_pct = p.pen_a != 0 ? 130 : 100;
    return launch_tc<2>(tq, tk, tks, p, p.n_groups * p.NQT, bf16, s.head_dim, st);
  }
  return launch_tc<0>(tq, tk, tk, p, p.n_groups * p.NQT, bf16, s.head_dim, st);
}

cudaError_t launch_fam_tc(const void* q, const void* k, const float* lse, int dtype, AttnShape s,
                          float scale, int window, float* F, void* ws, size_t ws_bytes, int* status,
                          cudaStream_t st, int per_head, const TargetOut* tgt) {
  const FamSched f = fam_schedule(s, window);
  if (ws_bytes < fam_tc_workspace_size(s, window, per_head)) return cudaErrorInvalidValue;
  TcParams p{};
  p.S = s.seq_len;
  p.Hq = s.h_q;
  p.Hkv = s.h_kv;
  p.G = s.h_q / s.h_kv;
  p.c2 = scale * KVP_LOG2E;
  p.inv_scale = 1.0f / scale;
  p.window = window;
  p.lse = lse;
  p.out = (float*)ws;
  p.n_groups = s.n_batch * s.h_kv;
  // Items in blocks of KV-head groups whose query rows together stay within about 96 MB of L2
  // (8 groups at S = 8192; 2 at S = 32768 and 1 at S = 131072 with G = 4: the 32-layer pass
  // 117.5 -> 115.5 ms and the 131072-token pass 54 -> 51 ms against blocks of 8).
  {
    const double q_group = (double)p.G * s.seq_len * s.head_dim * 2;
    const int gb = std::max(1, std::min(8, (int)(96e6 / q_group)));
    p.gblk = std::min(p.n_groups, gb);
  }
  p.NT0 = f.NT0;
  p.TPC = f.TPC;
  p.CMAX = f.CMAX;
  p.NKT = f.NKT;
  p.Nf = f.Nf;
  p.per_head = per_head;
  p.status = status;
  const long long items = (long long)(f.Nf + f.Np) * p.n_groups;
  if (items > 0) {
    const int BHq = s.n_batch * s.h_q, S_pad = s.seq_len + BN;
    void* ext = (char*)ws + fam_partial_bytes(s, f, per_head);
    int* queue = (int*)((char*)ext + fam_ext_bytes(s));
    CUtensorMap tq, tk, te;
    if (!make_q_tmap(&tq, q, dtype, s) || !make_k_tmap(&tk, k, dtype, s) ||
        !make_ext_tmap(&te, ext, dtype, BHq, S_pad))
      return cudaErrorInvalidValue;
    if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long rows = (long long)BHq * S_pad;
    long long blocks = (rows + 255) / 256;
    if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
    count_launches(1);
    cudaError_t e = launch_with_pdl(ext_prep_kernel, dim3((unsigned)blocks), dim3(256), 0, st, lse, BHq,
                                    s.seq_len, S_pad, p.inv_scale, dtype == KVP_BF16, (uint4*)ext, queue);
    if (e != cudaSuccess) return e;
    p.queue = queue;
    p.total_items = (int)items;
    e = s.head_dim == 64 ? launch_mass_persistent_hd<64>(tq, tk, te, p, dtype == KVP_BF16, st)
                         : launch_mass_persistent_hd<128>(tq, tk, te, p, dtype == KVP_BF16, st);
    if (e != cudaSuccess) return e;
  }
  count_launches(1);
  if (per_head) {                          // the per-head sums (and the target when asked for)
    const TargetOut none{0.f, 0, nullptr, nullptr};
    const TargetOut* t = tgt ? tgt : &none;
    return launch_with_pdl(fam_target_kernel, dim3(f.NKT, p.n_groups), dim3(BM), 0, st, (const float*)ws,
                           s.seq_len, s.h_kv, p.G, f.NT0, f.TPC, f.CMAX, f.NKT, window, t->eps, t->aggregate,
                           F, t->target, t->F);
  }
  return launch_with_pdl(fam_reduce_kernel, dim3(f.NKT, p.n_groups), dim3(BM), 0, st, (const float*)ws, s.seq_len,
                         f.NT0, f.TPC, f.CMAX, f.NKT, F);
}

}  // namespace kvp
