// Host-side launchers of libkvp's kernels (one translation unit each); called
// by kvp_abi.cu after argument validation.  Each returns cudaGetLastError().
#pragma once

#include <cuda_runtime.h>

#include <utility>
#include <stddef.h>
#include <stdint.h>

namespace kvp {

// Host-side count of kernel launches made by the library (diagnostics).
void count_launches(int n);

// Launch attribute that lets a kernel start while the previous kernel of its stream finishes
// (programmatic dependent launch); the kernel must call wait_prior_grid() before it touches
// global memory.
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a{};
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// Launches `kern` with programmatic dependent launch (the kernel must call wait_prior_grid()
// before it reads what the previous kernel of the stream wrote, or writes what it reads).
template <typename... KArgs, typename... Args>
cudaError_t launch_with_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Shape of a row-LSE / future-mass problem and the element strides of Q and K (batch, head,
// token; the head_dim axis is contiguous).  Dense [n_batch, H, S, D] tensors have strides
// (H*S*D, S*D, D).
struct AttnShape {
  int n_batch, h_q, h_kv, seq_len, head_dim;
  int64_t q_sb, q_sh, q_sr;
  int64_t k_sb, k_sh, k_sr;
};
inline AttnShape dense_attn_shape(int n_batch, int h_q, int h_kv, int S, int D) {
  const int64_t sd = (int64_t)S * D;
  return AttnShape{n_batch, h_q, h_kv, S, D, sd * h_q, sd, D, sd * h_kv, sd, D};
}

// Running top-k mask of the sparse row LSE: static ranks and cutoffs [n_batch*h_kv, S].
struct SparseMask {
  const int32_t* ranks;
  const int32_t* tau;
  int n_sink, window;
  // Tensor-core path only (null: dense streaming): workspace for the rank-ordered key stream --
  // the inverse permutation [n_batch*h_kv, S], the keys in rank order, a validity flag.
  int32_t* inv = nullptr;
  void* k_sorted = nullptr;
  int* perm_ok = nullptr;
};
// Workspace of the sparse row LSE on the tensor-core path (0 for the fp32 path).
size_t sparse_lse_workspace_size(int dtype, AttnShape s);

// fp32-FFMA tiled passes: the path for float32 inputs.  mask != null: the sparse row LSE.
cudaError_t launch_lse_simt(const void* q, const void* k, int dtype, AttnShape s, float scale,
                            float* lse, cudaStream_t st, const SparseMask* mask = nullptr);
cudaError_t launch_fam_simt(const void* q, const void* k, const float* lse, int dtype, AttnShape s,
                            float scale, int window, float* F, cudaStream_t st, int per_head = 0);
// KVpop target from per-query-head mass: count normalisation, log(eps + m), group max / mean.
cudaError_t launch_target_epilogue(const float* F_heads, int n_batch, int h_q, int h_kv, int S,
                                   int window, float eps, int aggregate, float* target, float* F,
                                   cudaStream_t st);

// tcgen05 / TMA passes (bf16 / f16, head_dim 64 or 128).  tc_encoder_available() is false when
// the driver's tensor-map encoder cannot be resolved (then these passes cannot run).
bool tc_encoder_available();
size_t fam_tc_workspace_size(AttnShape s, int window, int per_head = 0);
// mask == null: the dense row LSE; mask != null: the sparse row LSE.
cudaError_t launch_lse_tc(const void* q, const void* k, int dtype, AttnShape s, float scale,
                          float* lse, int* status, cudaStream_t st, const SparseMask* mask = nullptr);
// KVpop target outputs computed straight from the per-head partial sums (per_head = 1): N_t,
// log(eps + m), group max or probability-space mean; target and F nullable.
struct TargetOut {
  float eps;
  int aggregate;
  float* target;   // [n_batch, h_kv, seq_len]
  float* F;        // [n_batch, h_kv, seq_len]
};
// per_head = 1: F receives each query head's mass, [n_batch, h_q, seq_len] (nullable when tgt is
// given).
cudaError_t launch_fam_tc(const void* q, const void* k, const float* lse, int dtype, AttnShape s,
                          float scale, int window, float* F, void* ws, size_t ws_bytes,
                          int* status, cudaStream_t st, int per_head = 0, const TargetOut* tgt = nullptr);

cudaError_t launch_soft_topk(const double* x, int n, double k, int t, double* ratios,
                             int32_t* budgets, cudaStream_t st);
// scores_b != null: the row is scores[0, n_a) followed by scores_b[0, T - n_a).
// budgets == null: every row's budget is b_uniform.
cudaError_t launch_select(const float* scores, int R, int T, int64_t row_stride,
                          const int32_t* budgets, int n_sink, int n_recent, int32_t* idx,
                          int b_max, int32_t* count, int* status, cudaStream_t st,
                          const float* scores_b = nullptr, int64_t row_stride_b = 0, int n_a = 0,
                          int b_uniform = 0);
cudaError_t launch_compact(const void* k, const void* v, int row_bytes, int R, int T,
                           const int32_t* idx, const int32_t* count, int b_max, void* k_out,
                           void* v_out, int* status, cudaStream_t st);
// Chunked prefill-compress: gather kept entries of [cache (n_in per row) ; chunk (C per row)]
// -- K, V rows, scores and source positions -- into the output cache (row capacity out_cap).
struct ChunkSrc {
  const void* cache_k;
  const void* cache_v;
  const float* cache_score;
  const int32_t* cache_pos;
  int cap_in, n_in;
  const void* chunk_k;
  const void* chunk_v;
  const float* chunk_score;
  int C, pos0;
};
cudaError_t launch_chunk_compact(const ChunkSrc& src, int row_bytes, int R, const int32_t* idx,
                                 const int32_t* count, int b_max, void* out_k, void* out_v,
                                 float* out_score, int32_t* out_pos, int out_cap, int* status,
                                 cudaStream_t st);

// Running top-k cutoffs tau [n_heads, S] from static ranks (a permutation of 0..S-1 per head).
cudaError_t launch_topk_cutoffs(const int32_t* ranks, int n_heads, int S, int n_sink, int window,
                                int k, int32_t* tau, int* status, cudaStream_t st);

// Per-row ranks of scores (0 = highest, ties to the lower index, NaN last) and the
// eviction-cost AUC sum_t (rank_t + 1) * F_t of M rankings per row.
size_t rank_rows_workspace_size(int R, int T);
cudaError_t launch_rank_rows(const float* scores, int R, int T, int32_t* ranks, void* ws,
                             int* status, cudaStream_t st);
size_t eviction_auc_workspace_size(int R, int M, int T);
cudaError_t launch_eviction_auc(const float* F, const int32_t* ranks, int R, int M, int T,
                                double* auc, void* ws, cudaStream_t st);

cudaError_t launch_ring_insert(void* kc, void* vc, int32_t* slot_pos, float* slot_score, int32_t* fill,
                               int R, int cap, int row_bytes, const void* new_k, const void* new_v,
                               int new_pos, int n_sink, int n_recent, int32_t* out_slot, int* status,
                               cudaStream_t st);

struct DecodePlan {
  int R, G;
  // fp32 cache path (grid of key chunks x rows)
  int n_chunks, chunk;
  size_t partial_bytes, lse_bytes, logit_bytes, simt_total_bytes;
  // bf16/f16 cache path (persistent stream-K CTAs over 64-key tiles)
  int nt, n_ctas, maxseg;
  int lg_smem_keys;     // > 0: the key-mass logits of a CTA stay in shared memory (keys per CTA)
  size_t mma_partial_bytes, counter_bytes, mma_lse_bytes, mma_logit_bytes, mma_total_bytes;
  size_t total_bytes;   // workspace that covers either path
};
void decode_mma_plan(DecodePlan& p, int head_dim, int T_cap, int with_key_mass);
cudaError_t launch_decode_mma(const void* q, const void* kc, const void* vc, int dtype, int n_layers,
                              int h_q, int h_kv, int head_dim, int T_cap, const int32_t* len,
                              float scale, float* out, float* key_mass, const int32_t* key_pos,
                              int T_src, int accumulate, const DecodePlan& plan, void* ws,
                              int* status, cudaStream_t st);
DecodePlan decode_plan(int n_layers, int h_q, int h_kv, int head_dim, int T_cap, int with_key_mass);
// Static scratch of kvp_decode_attn_noalloc on the current device (set up on first use, and
// again in a new context of the device).  _ready(): the address is already cached for the
// current context.
bool decode_noalloc_scratch_ready();
cudaError_t decode_noalloc_scratch(void** ptr, size_t* bytes);
// The calling thread's current CUDA context (a CUcontext; null when none is current or the
// driver entry point cannot be resolved).  Keys the cached device addresses of the library's
// static symbols.
void* current_cu_context();
cudaError_t launch_decode(const void* q, const void* kc, const void* vc, int dtype, int n_layers,
                          int h_q, int h_kv, int head_dim, int T_cap, const int32_t* len,
                          float scale, float* out, float* key_mass, const int32_t* key_pos,
                          int T_src, int accumulate, const DecodePlan& plan, void* ws,
                          int* status, cudaStream_t st);

}  // namespace kvp
