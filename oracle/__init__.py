"""Plain, slow, fp64 CPU oracle of the future-attention-mass / pruned-cache path.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import it.  It shares no code with
the CUDA library (``learned_kv_cache_gb300``) and neither imports the other; the
seeded inputs come from ``kvp_inputs``.

Functions and the passages they follow:

* :func:`row_lse`, :func:`future_attn_mass`, :func:`future_attn_mass_per_head`,
  :func:`kvpop_target` -- KVpop, "Defining Future Attention Utility", "Delayed
  Memory Scoring", "Alternative Aggregation Methods" and Figure 2.
* :func:`select_topk`, :func:`compact_kv` -- KVpop "The KVpop Scoring Module";
  Learning to Evict from Key-Value Cache §1, §4.1, §A.2; How much KV cache can
  you prune, "What we did" and "Conclusion".
* :func:`decode_attn` -- How much KV cache can you prune, "Bounded windows".
* :func:`ring_victim`, :func:`ring_insert` -- How much KV cache can you prune,
  "What we did" and "Conclusion" (static cache overwritten in place).
* :func:`rank_by_scores`, :func:`eviction_cost_curve`, :func:`eviction_auc`,
  :func:`optimal_auc`, :func:`normalized_auc` -- Learning to Evict from Key-Value Cache §1, §3
  and §3.1.1 (a ranking serves every budget; cost-versus-budget area under the curve,
  normalised by the optimal ranking).
* :func:`chunk_compress_step`, :func:`chunked_prefill_compress` -- Learning to Evict from
  Key-Value Cache §4 and §4.1 (chunked prefill-compress with physical compaction).
* :func:`fenwick_cutoffs`, :func:`sparse_mask`, :func:`sparse_row_lse` -- KVpop, "Efficient
  Online Pruning", "Fenwick-tree cut-off computation (Algorithm 2)" and "Delayed Memory
  Scoring" (the sparse log-normalisers).
* :func:`soft_topk`, :func:`head_budgets` -- LKV, "The Differentiable Soft-TopK
  Operator" and "LKV-H".

Every function is pinned by the ``-m "not gpu"`` tests (brute force through
library softmax/logsumexp on tiny inputs, closed forms, invariants and the
pages' worked examples).
"""
from .attention_mass import future_attn_mass, future_attn_mass_per_head, kvpop_target, row_lse
from .budgets import head_budgets, soft_topk
from .decode import decode_attn
from .auc import eviction_auc, eviction_cost_curve, normalized_auc, optimal_auc, rank_by_scores
from .chunked import chunk_compress_step, chunked_prefill_compress
from .fenwick import fenwick_cutoffs, sparse_mask, sparse_row_lse
from .ring import ring_insert, ring_victim
from .selection import compact_kv, effective_budget, select_row, select_topk

__all__ = [
    "row_lse", "future_attn_mass", "future_attn_mass_per_head", "kvpop_target", "select_topk", "select_row", "effective_budget",
    "compact_kv", "decode_attn", "soft_topk", "head_budgets", "ring_insert", "ring_victim",
    "fenwick_cutoffs", "sparse_mask", "sparse_row_lse", "chunk_compress_step", "chunked_prefill_compress",
    "rank_by_scores", "eviction_cost_curve", "eviction_auc", "optimal_auc", "normalized_auc",
]
