/*
 * kvp.h -- C ABI of the future-attention-mass / pruned-KV-cache hot path (sm_103a).
 *
 * Five stages, one entry point each, plus the head-wise budget helper:
 *
 *   kvp_lse_pass           causal row log-sum-exp of the attention logits
 *   kvp_future_attn_mass   transposed (key-major) pass: future-attention mass per key
 *   kvp_soft_topk_budgets  closed-form Soft-TopK head ratios and budgets b = floor(r * t)
 *   kvp_select_topk        sinks + recent window + top-k fill under per-row budgets
 *   kvp_compact_kv         gather of the kept K/V rows into a dense pruned cache
 *   kvp_decode_attn        one-token decode attention over the (pruned) cache
 *
 * and the steps either side of them: kvp_future_attn_target (KVpop's supervision
 * target), kvp_ring_insert (in-place eviction of a static decode cache),
 * kvp_chunk_compress (one step of chunked prefill-compress), kvp_rank_rows and
 * kvp_eviction_auc (static ranks; KVP's eviction-cost area of a ranking),
 * kvp_topk_cutoffs and kvp_sparse_lse_pass (KVpop's running top-k sparse
 * attention and its log-normalisers).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer argument is a DEVICE pointer unless stated otherwise; the
 *   caller owns all buffers.  The library never allocates, frees or
 *   synchronises (except kvp_check_device_status, which synchronises the given
 *   stream).  Work is enqueued asynchronously on `stream` (a cudaStream_t;
 *   NULL = the legacy default stream).
 * - Arguments are validated on the host before anything is launched; a call
 *   that returns an error has enqueued nothing.  Errors that only the device
 *   can see (an out-of-range index or budget in a device array, a bounded wait
 *   that gave up) are recorded in a per-device status word that
 *   kvp_check_device_status() reads and clears; the affected outputs are then
 *   unspecified.
 * - Tensors are row-major with the last dimension contiguous; the layout of
 *   each argument is given in brackets.  They are dense unless the entry point
 *   takes strides (the Q/K inputs of the attention passes).  Q/K/V base
 *   pointers must be 16-byte aligned.
 * - head_dim must be 64 or 128.  Logits are scaled by `sm_scale` (normally
 *   1/sqrt(head_dim)); all softmax arithmetic is fp32.
 * - GQA: query head h_q belongs to KV head h_q / (h_q_count / h_kv_count).
 */
#ifndef KVP_H
#define KVP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVP_ABI_VERSION 2

/* A cudaStream_t (struct CUstream_st*), declared without pulling in CUDA headers. */
typedef struct CUstream_st* kvp_stream_t;

typedef enum kvp_dtype {
  KVP_F32 = 0,  /* float32 */
  KVP_BF16 = 1, /* bfloat16 */
  KVP_F16 = 2   /* IEEE half */
} kvp_dtype;

typedef enum kvp_status {
  KVP_OK = 0,
  KVP_ERR_INVALID_ARG = -1,   /* null pointer, bad size, misaligned buffer, ... */
  KVP_ERR_UNSUPPORTED = -2,   /* dtype / head_dim / layout this build does not handle */
  KVP_ERR_CUDA = -3,          /* a CUDA runtime call failed; see kvp_last_error() */
  KVP_ERR_TIMEOUT = -4,       /* device status: a bounded wait inside a kernel gave up */
  KVP_ERR_WORKSPACE = -5,     /* workspace pointer null or smaller than the size query */
  KVP_ERR_DEVICE_CHECK = -6   /* device status: a device-side index/budget was out of range */
} kvp_status;

/* ---------------------------------------------------------------------------
 * Q / K strides of the attention passes (kvp_lse_pass, kvp_sparse_lse_pass,
 * kvp_future_attn_mass, kvp_future_attn_target).
 *
 * q_strides / k_strides are HOST arrays of three int64 element strides
 * {batch, head, token} of q and k (the head_dim axis is always contiguous), or
 * NULL for the dense layout [n_batch, H, seq_len, head_dim].  A slice of a
 * fused QKV projection [seq_len, (h_q + 2 h_kv) * head_dim] is read in place
 * with q_strides = {-, head_dim, (h_q + 2 h_kv) * head_dim}.  Every stride
 * that is used must be a positive multiple of 16 bytes below 2^40 bytes, the
 * token stride at least head_dim; the stride of an extent-1 dimension (batch
 * when n_batch = 1, head when there is one head) is ignored.  Outputs (lse, F,
 * target, F_heads) are always dense.
 *
 * Paths: bf16 / f16 inputs run on the tcgen05 tensor-core passes (head_dim 64
 * or 128, operands loaded by TMA); float32 inputs on the fp32-FFMA passes.
 * There is no other path: when the driver's tensor-map encoder cannot be
 * resolved, 16-bit calls fail with KVP_ERR_CUDA.
 * ------------------------------------------------------------------------- */

/* ---------------------------------------------------------------------------
 * A1. Causal row log-sum-exp.
 *
 * KVpop -- Key-Value Cache Compression with Predictive Online Pruning,
 * "Delayed Memory Scoring" (worked LSE example) and Figure 2: the per-query
 * log-normaliser that attention kernels return as their auxiliary LSE.
 *
 *   lse[b, h, i] = ln sum_{j <= i} exp(sm_scale * q[b, h, i, :] . k[b, h / G, j, :])
 *
 * q   [n_batch, h_q,  seq_len, head_dim]  dtype
 * k   [n_batch, h_kv, seq_len, head_dim]  dtype
 * lse [n_batch, h_q,  seq_len]            float32, natural log (output)
 * n_batch counts independent problems (e.g. layers).  bf16/f16 inputs run on
 * the tensor cores (fp32 accumulation); float32 inputs on fp32 FFMA.
 * q_strides / k_strides: see "Q / K strides" above (NULL = dense).
 * ------------------------------------------------------------------------- */
int kvp_lse_pass(const void* q, const void* k, int dtype, int n_batch, int h_q, int h_kv,
                 int seq_len, int head_dim, const int64_t* q_strides, const int64_t* k_strides,
                 float sm_scale, float* lse, kvp_stream_t stream);

/* ---------------------------------------------------------------------------
 * A2. Future-attention mass (transposed, key-major column pass).
 *
 * KVpop, "Defining Future Attention Utility", "Delayed Memory Scoring" and
 * Figure 2: the attention mass key j receives from the queries that have
 * left the protected window (i >= j + window), obtained by swapping the roles
 * of queries and keys and offsetting each logit by the query's LSE; summed
 * over the GQA group of the KV head (raw sum: no count normalisation, no log):
 *
 *   F[b, h, j] = sum_{g < G} sum_{i = j + window}^{seq_len - 1}
 *                exp(sm_scale * q[b, h*G+g, i] . k[b, h, j] - lse[b, h*G+g, i])
 *
 * The S x S matrix is never formed.  Keys j > seq_len - 1 - window get 0.
 * q, k (and their strides) as in kvp_lse_pass; lse is kvp_lse_pass's output.
 * F [n_batch, h_kv, seq_len] float32 (output).
 * workspace: device scratch of at least kvp_future_attn_mass_workspace_size()
 * bytes (partial sums, the query-side LSE operand, a work counter; may be NULL
 * when that size is 0).  Calls that run at the same time need separate
 * workspaces.
 * ------------------------------------------------------------------------- */
size_t kvp_future_attn_mass_workspace_size(int dtype, int n_batch, int h_q, int h_kv,
                                           int seq_len, int head_dim, int window);
int kvp_future_attn_mass(const void* q, const void* k, const float* lse, int dtype, int n_batch,
                         int h_q, int h_kv, int seq_len, int head_dim, const int64_t* q_strides,
                         const int64_t* k_strides, float sm_scale, int window, float* F,
                         void* workspace, size_t workspace_bytes, kvp_stream_t stream);

/* ---------------------------------------------------------------------------
 * A2'. KVpop's supervision target (per-query-head future mass and its epilogue).
 *
 * KVpop, "Defining Future Attention Utility" (count normalisation N_t =
 * max(1, S - (t + w)), the mean m_g(t) = F_g(t) / N_t of every query head g,
 * log(eps + m) and the max over the heads that share a KV head; worked example
 * N_t = 2, means 0.25 / 0.10, target -1.386) and "Alternative Aggregation
 * Methods" (the probability-space mean over the group):
 *
 *   F_g[b, h*G+g, t] = sum_{i = t + window}^{seq_len - 1}
 *                      exp(sm_scale * q[b, h*G+g, i] . k[b, h, t] - lse[b, h*G+g, i])
 *   KVP_TARGET_MAX_LOG:   target[b, h, t] = max_g log(eps + F_g / N_t)
 *   KVP_TARGET_MEAN_PROB: target[b, h, t] = log(eps + (1/G) sum_g F_g / N_t)
 *
 * Inputs (and strides) as in kvp_future_attn_mass.  Outputs (each nullable, at least one):
 * target [n_batch, h_kv, seq_len] float32; F_heads [n_batch, h_q, seq_len]
 * float32 (the per-query-head mass); F [n_batch, h_kv, seq_len] float32 (their
 * group sum).  eps >= 0 (eps = 0 gives -inf where a key receives no mass);
 * sm_scale > 0.  workspace: at least kvp_future_attn_target_workspace_size()
 * bytes, 256-byte aligned.
 * ------------------------------------------------------------------------- */
#define KVP_TARGET_MAX_LOG 0
#define KVP_TARGET_MEAN_PROB 1
size_t kvp_future_attn_target_workspace_size(int dtype, int n_batch, int h_q, int h_kv,
                                             int seq_len, int head_dim, int window);
int kvp_future_attn_target(const void* q, const void* k, const float* lse, int dtype, int n_batch,
                           int h_q, int h_kv, int seq_len, int head_dim, const int64_t* q_strides,
                           const int64_t* k_strides, float sm_scale, int window, float eps,
                           int aggregate, float* target, float* F_heads, float* F, void* workspace,
                           size_t workspace_bytes, kvp_stream_t stream);

/* ---------------------------------------------------------------------------
 * A1'. Running top-k cutoffs (KVpop's online pruning during prefill/training).
 *
 * KVpop, "Efficient Online Pruning" and "Fenwick-tree cut-off computation
 * (Algorithm 2)": every token of a KV head has a static rank (0 = most
 * important; a permutation of 0..seq_len-1 per head).  At query q the token
 * t = q - window leaves the protected window and becomes eligible unless
 * t < n_sink.  Once k tokens are eligible, tau[h, q] is the k-th smallest rank
 * among the eligible tokens (the rank threshold of the top-k eligible set);
 * before that tau[h, q] = -1.  The page keeps the eligible ranks in a Fenwick
 * tree; this library computes the same thresholds with per-chunk bitmaps.
 *
 * ranks [n_heads, seq_len] int32 (input), tau [n_heads, seq_len] int32 (output).
 * 1 <= seq_len <= 524288, k >= 1, n_sink >= 0, window >= 0.  Ranks that are
 * out of range or repeated are reported through the device status
 * (KVP_ERR_DEVICE_CHECK) and leave tau unspecified.
 * ------------------------------------------------------------------------- */
int kvp_topk_cutoffs(const int32_t* ranks, int n_heads, int seq_len, int n_sink, int window,
                     int k, int32_t* tau, kvp_stream_t stream);

/* ---------------------------------------------------------------------------
 * A1''. Sparse row log-sum-exp (the student's log-normalisers).
 *
 * KVpop, "Efficient Online Pruning" (query q attends to the sink tokens, the
 * protected window and the eligible tokens of rank <= tau_q) and "Delayed
 * Memory Scoring" (the future-attention target reuses these sparse
 * log-normalisers; pass the result as `lse` to kvp_future_attn_mass or
 * kvp_future_attn_target):
 *
 *   keep(i, j) = j <= i and (j < n_sink or j > i - window or tau[i] < 0 or rank[j] <= tau[i])
 *   lse[b, h, i] = ln sum_{j : keep(i, j)} exp(sm_scale * q[b, h, i] . k[b, h/G, j])
 *
 * tau[i] < 0 (fewer than k eligible tokens) keeps every eligible token.
 * q, k (and strides), lse as in kvp_lse_pass; ranks and tau [n_batch, h_kv, seq_len] int32
 * (kvp_topk_cutoffs' input and output; any int32 values are accepted, the
 * mask is applied as written).  workspace: kvp_sparse_lse_workspace_size()
 * bytes, 256-byte aligned (0 for the fp32 path).  On the tensor-core path a
 * query tile whose rows all have a cutoff streams, instead of every causal
 * key tile, the tiles holding its sinks and windows plus the keys in rank
 * order up to the largest cutoff of its rows (the workspace holds the inverse
 * permutation and the keys in rank order), whenever that is fewer tiles;
 * ranks that are not a permutation fall back to the dense stream.
 * ------------------------------------------------------------------------- */
size_t kvp_sparse_lse_workspace_size(int dtype, int n_batch, int h_q, int h_kv, int seq_len,
                                     int head_dim);
int kvp_sparse_lse_pass(const void* q, const void* k, const int32_t* ranks, const int32_t* tau,
                        int dtype, int n_batch, int h_q, int h_kv, int seq_len, int head_dim,
                        const int64_t* q_strides, const int64_t* k_strides, float sm_scale,
                        int n_sink, int window, float* lse, void* workspace, size_t workspace_bytes,
                        kvp_stream_t stream);

/* ---------------------------------------------------------------------------
 * Ranks of score rows (static ranks; the optimal ranking of the eviction cost).
 *
 * KVpop, "Efficient Online Pruning" (tokens are pre-sorted by a static priority
 * score and their ranks stored, for kvp_topk_cutoffs) and Learning to Evict
 * from Key-Value Cache §3.1.1 (the optimal ranking orders entries by their
 * importance):
 *
 *   ranks[r, t] = position of entry t when row r is sorted by score, highest
 *                 first; equal scores in index order; NaN last; -0.0 == +0.0
 *
 * scores [R, T] float32, ranks [R, T] int32 (output, a permutation of 0..T-1
 * per row).  workspace: kvp_rank_rows_workspace_size(R, T) bytes, 256-byte
 * aligned (radix-sort buffers).  R <= 65535.
 * ------------------------------------------------------------------------- */
size_t kvp_rank_rows_workspace_size(int R, int T);
int kvp_rank_rows(const float* scores, int R, int T, int32_t* ranks, void* workspace,
                  size_t workspace_bytes, kvp_stream_t stream);

/* ---------------------------------------------------------------------------
 * Eviction-cost area under the curve of a ranking (KVP's global reward).
 *
 * Learning to Evict from Key-Value Cache §1, §3 and §3.1.1: one ranking serves
 * every budget b (entries of rank < b are kept); cost(b) is the importance of
 * the entries it evicts, and the ranking is scored by the area under cost(b)
 * over all budgets, normalised by the optimal ranking's area:
 *
 *   auc[r, m] = sum_{b=0}^{T} sum_{t : ranks[r,m,t] >= b} F[r, t]
 *             = sum_t (ranks[r, m, t] + 1) * F[r, t]
 *
 * F [R, T] float32 (e.g. kvp_future_attn_mass's output), ranks [R, M, T] int32
 * (M rankings per row, each taken as given), auc [R, M] float64 (output).  The
 * normalised cost of a ranking is its auc divided by the auc of
 * kvp_rank_rows(F).  Products and sums are exact to fp64 rounding.
 * workspace: kvp_eviction_auc_workspace_size(R, M, T) bytes (per-chunk partial
 * sums, added in fixed order).  R, M <= 65535 and R * M <= 2^24.
 * ------------------------------------------------------------------------- */
size_t kvp_eviction_auc_workspace_size(int R, int M, int T);
int kvp_eviction_auc(const float* F, const int32_t* ranks, int R, int M, int T, double* auc,
                     void* workspace, size_t workspace_bytes, kvp_stream_t stream);

/* ---------------------------------------------------------------------------
 * A0. Head-wise budgets from the closed-form Soft-TopK.
 *
 * LKV: End-to-End Learning of Head-wise Budgets and Token Selection for LLM
 * KV Cache Eviction, "The Differentiable Soft-TopK Operator" (threshold
 * lambda in closed form over the descending-sorted scores) and "LKV-H"
 * (ratios r = ST_k(s) over the flattened head scores, budget b = floor(r*t)).
 * Each ratio is the Laplace CDF of (s_i - lambda), the map whose budget
 * equation sum_i r_i = k solves to the printed threshold; sum_i r_i = k.
 *
 * scores  [n] float64;  ratios [n] float64 (output);  budgets [n] int32 (output).
 * Requires 1 <= n <= 1024, 0 < k < n, t >= 0, scores finite with |s| < 700.
 * ------------------------------------------------------------------------- */
int kvp_soft_topk_budgets(const double* scores, int n, double k, int t, double* ratios,
                          int32_t* budgets, kvp_stream_t stream);

/* ---------------------------------------------------------------------------
 * A3. Budgeted per-row selection.
 *
 * KVpop, "The KVpop Scoring Module" and Figure 1 (sink tokens and a
 * protected recent window are always kept; the top-k scores fill the rest of
 * the fixed budget: 2 + 3 + 4 = 9 = B in its example); Learning to Evict from
 * Key-Value Cache, §1 and §A.2 (discard the lowest-ranked entries to meet the
 * budget; first four and last 16 always kept); How much KV cache can you
 * prune, "What we did" (keep the first four, the newest 32, fill the rest).
 *
 * For each row r of scores [R, row_stride] (first T entries used):
 *   b_eff = T if T <= b[r], else max(b[r], n_sink + n_recent);
 *   keep [0, n_sink) and [T - n_recent, T), then the k = b_eff - n_sink - n_recent
 *   highest scores of the middle, ties to the LOWER index, -0.0 == +0.0,
 *   NaN below -inf.
 * budgets [R] int32 (device);  idx [R, b_max] int32 (output): kept token
 * indices in ascending order, padded with -1;  count [R] int32 (output) = b_eff.
 * A row whose b_eff exceeds b_max (or whose budget is negative) gets
 * count = -1 and raises KVP_ERR_DEVICE_CHECK in the device status.
 * ------------------------------------------------------------------------- */
int kvp_select_topk(const float* scores, int R, int T, int64_t row_stride,
                    const int32_t* budgets, int n_sink, int n_recent, int32_t* idx,
                    int b_max, int32_t* count, kvp_stream_t stream);

/* ---------------------------------------------------------------------------
 * A4. Compaction of the kept entries into a dense pruned cache.
 *
 * Learning to Evict from Key-Value Cache, §4.1 (chunked prefill-compress with
 * physical tensor compaction); How much KV cache can you prune, "Conclusion"
 * (the kept entries are copied into a new tensor).  Byte copy:
 *
 *   k_out[r, m, :] = k[r, idx[r, m], :],  v_out likewise,  for m < count[r]
 *
 * k, v [R, T, head_dim] dtype;  idx [R, b_max], count [R] from kvp_select_topk;
 * k_out, v_out [R, b_max, head_dim] dtype (output; rows m >= count[r] are
 * not written).  An index outside [0, T) raises KVP_ERR_DEVICE_CHECK.
 * ------------------------------------------------------------------------- */
int kvp_compact_kv(const void* k, const void* v, int dtype, int R, int T, int head_dim,
                   const int32_t* idx, const int32_t* count, int b_max, void* k_out,
                   void* v_out, kvp_stream_t stream);

/* ---------------------------------------------------------------------------
 * A3'/A4''. One step of chunked prefill-compress.
 *
 * Learning to Evict from Key-Value Cache §4 and §4.1 (long contexts are
 * prefilled chunk by chunk and the cache is compressed back to the budget
 * after every chunk, with physical tensor compaction; budgets uniform across
 * heads and layers) with the selection rule of kvp_select_topk (sinks, the
 * most recent tokens and the top-scoring rest; scores are the per-token,
 * query-agnostic ranking scores that stay with a token while it is kept):
 *
 *   union[r] = cache[r, 0 .. n_in) followed by chunk[r, 0 .. chunk_len)
 *   kept     = kvp_select_topk(union scores, budget, n_sink, n_recent)
 *   out[r, m] = union[r, idx[r, m]]  (K, V rows, score, source position)
 *
 * cache_k, cache_v [R, cap_in, head_dim] dtype; cache_score [R, cap_in] float32;
 * cache_pos [R, cap_in] int32 (source positions): the previous step's output,
 * n_in entries valid per row (n_in = 0: the first chunk; the cache pointers
 * may then be null).  chunk_k, chunk_v [R, chunk_len, head_dim]; chunk_score
 * [R, chunk_len]; the chunk's source positions are pos0 .. pos0+chunk_len-1.
 * idx [R, out_cap] int32 (kept union indices, ascending, -1 padded) and
 * count [R] int32 (kept per row: min(n_in + chunk_len, max(budget,
 * n_sink + n_recent))) are outputs; so are out_k, out_v [R, out_cap,
 * head_dim], out_score [R, out_cap], out_pos [R, out_cap] (the next step's
 * cache; the output must not alias the inputs).  out_cap >= the kept count.
 * ------------------------------------------------------------------------- */
int kvp_chunk_compress(const void* cache_k, const void* cache_v, const float* cache_score,
                       const int32_t* cache_pos, int cap_in, int n_in, const void* chunk_k,
                       const void* chunk_v, const float* chunk_score, int chunk_len, int pos0,
                       int dtype, int R, int head_dim, int budget, int n_sink, int n_recent,
                       int32_t* idx, int32_t* count, void* out_k, void* out_v, float* out_score,
                       int32_t* out_pos, int out_cap, kvp_stream_t stream);

/* ---------------------------------------------------------------------------
 * A4'. In-place eviction of a static (ring) decode cache.
 *
 * How much KV cache can you prune, "What we did" (attention-score policy: keep
 * the first tokens, always keep the newest ones, fill the rest with the tokens
 * that received the most attention) and "Conclusion" (a ring or static cache
 * overwrites old entries in place instead of copying the kept ones).
 *
 * Per row r of a cache with `cap` slots: if fill[r] < cap the new token is
 * appended at slot fill[r] and fill[r] grows by one; otherwise the slot with the
 * lowest slot_score among the slots whose token position p satisfies
 * n_sink <= p <= new_pos - n_recent is overwritten (NaN first, -0.0 == +0.0,
 * ties to the newer token).  The chosen slot receives new_k / new_v, position
 * new_pos and score 0; out_slot[r] (nullable) reports it.
 *
 * kc, vc [R, cap, head_dim] dtype (updated in place); slot_pos [R, cap] int32;
 * slot_score [R, cap] float32 (the cumulative attention each slot's token has
 * received, e.g. accumulated by kvp_decode_attn's key mass with key_pos NULL);
 * fill [R] int32; new_k, new_v [R, head_dim] dtype.  Requires
 * cap >= n_sink + n_recent and n_recent >= 1 (then a full cache always has a
 * slot to give up); positions in a full row must be distinct, else
 * KVP_ERR_DEVICE_CHECK.
 * ------------------------------------------------------------------------- */
int kvp_ring_insert(void* kc, void* vc, int32_t* slot_pos, float* slot_score, int32_t* fill,
                    int dtype, int R, int cap, int head_dim, const void* new_k, const void* new_v,
                    int new_pos, int n_sink, int n_recent, int32_t* out_slot, kvp_stream_t stream);

/* ---------------------------------------------------------------------------
 * A5. Single-token decode attention over a (pruned) cache, split along keys.
 *
 * How much KV cache can you prune, "What we did" and "Bounded windows"
 * (one-token attention over the retained entries); KVpop Figure 1
 * (attention is computed over the retained set):
 *
 *   out[l, h, :] = sum_{m < len[r]} softmax_m(sm_scale * q[l, h] . kc[r, m]) vc[r, m],
 *   r = l * h_kv + h / G;  len[r] = 0 gives a zero output.
 *
 * q [n_layers, h_q, head_dim] dtype;  kc, vc [n_layers*h_kv, T_cap, head_dim] dtype;
 * len [n_layers*h_kv] int32 (device, each in [0, T_cap], else
 * KVP_ERR_DEVICE_CHECK);  out [n_layers, h_q, head_dim] float32 (output).
 * Optional key mass (key_mass != NULL): the probability each retained key
 * receives, summed over the group's query heads (the cumulative past-attention
 * score of the attention-score policy in How much KV cache can you prune), is
 * written (accumulate = 0: the whole [R, T_src] array is overwritten, zeros
 * where no retained key maps) or added (accumulate = 1) to
 * key_mass [R, T_src] float32 at position key_pos[r, m] ([R, T_cap] int32,
 * in [0, T_src)) or at m when key_pos is NULL (then T_src >= T_cap).
 * Requires G = h_q / h_kv <= 8.
 * workspace: at least kvp_decode_attn_workspace_size() bytes.
 * ------------------------------------------------------------------------- */
size_t kvp_decode_attn_workspace_size(int n_layers, int h_q, int h_kv, int head_dim, int T_cap,
                                      int with_key_mass);
int kvp_decode_attn(const void* q, const void* kc, const void* vc, int dtype, int n_layers,
                    int h_q, int h_kv, int head_dim, int T_cap, const int32_t* len,
                    float sm_scale, float* out, float* key_mass, const int32_t* key_pos,
                    int T_src, int accumulate, void* workspace, size_t workspace_bytes,
                    kvp_stream_t stream);

/* ---------------------------------------------------------------------------
 * A5 without a workspace: kvp_decode_attn_noalloc.
 *
 * Not a step of the method -- the pages have no counterpart.  It exists for
 * callers that cannot hand the library a workspace: programs whose device
 * memory is already fully reserved by their own pool (an inference server
 * that carved HBM into its KV cache), plain-C hosts with no device allocator
 * of their own, and decode loops that must not call cudaMalloc/cudaFree,
 * which can synchronise the whole device and stall work on other streams.
 *
 * Same computation, arguments and output as kvp_decode_attn without the key
 * mass (no key_mass / key_pos / T_src / accumulate) and without the
 * workspace: the split-K partials go to a fixed scratch array of
 * KVP_DECODE_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that
 * loads the library holds until the process exits.  A shape whose partials
 * need more than that is rejected with KVP_ERR_WORKSPACE (and a message
 * naming both sizes) before anything is launched.  The call allocates
 * nothing and calls no allocating routine.
 *
 * - The first call on each device looks up the scratch array's device
 *   address (a CUDA runtime query, cached per device and CUDA context); make
 *   that first call before capturing any stream on that device.  A first call
 *   made on a capturing stream is refused with KVP_ERR_INVALID_ARG.
 * - With lazy module loading (the CUDA default), that first lookup may be the
 *   moment the library's device code is loaded on the device, and with it the
 *   fixed array is placed in device memory: the driver's module load, not a
 *   cudaMalloc by the library, and once per device and context.  After
 *   cudaDeviceReset the next call runs in a new context and looks the address
 *   up again.
 * - All calls on a device share the one array and it keeps the last call's
 *   contents.  Each call clears, on its stream, what must start at zero (the
 *   per-row merge counters of the split-K path); every partial is written
 *   before it is read.  Calls whose executions overlap on the GPU (different
 *   streams, or host threads without ordering) race on the scratch and
 *   produce wrong outputs: serialise them, e.g. on one stream.
 * ------------------------------------------------------------------------- */
#define KVP_DECODE_NOALLOC_SCRATCH_BYTES (8u << 20) /* 8 MiB per device */
int kvp_decode_attn_noalloc(const void* q, const void* kc, const void* vc, int dtype, int n_layers,
                            int h_q, int h_kv, int head_dim, int T_cap, const int32_t* len,
                            float sm_scale, float* out, kvp_stream_t stream);

/* ---------------------------------------------------------------------------
 * Status and diagnostics.
 * ------------------------------------------------------------------------- */
/* Static string for a kvp_status code. */
const char* kvp_status_string(int status);
/* Message of the last failing call on this host thread ("" if none). */
const char* kvp_last_error(void);
/* Synchronises `stream`, then reads and clears the current device's status
 * word: KVP_OK, KVP_ERR_TIMEOUT or KVP_ERR_DEVICE_CHECK (first error recorded
 * since the last read), or KVP_ERR_CUDA if the synchronisation failed. */
int kvp_check_device_status(kvp_stream_t stream);
/* KVP_ABI_VERSION of the loaded library. */
int kvp_abi_version(void);
/* Number of kernels this process has launched through the library so far
 * (host-side counter, for accounting in benchmarks). */
uint64_t kvp_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* KVP_H */
