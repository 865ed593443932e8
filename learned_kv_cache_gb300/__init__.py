"""GB300-native future-attention mass and pruned KV cache.

The compute lives in ``libkvp.so`` (hand-written sm_103a CUDA kernels behind
the C ABI of ``include/kvp.h``); this package is its thin ctypes binding.
"""
from ._lib import (KVP_BF16, KVP_F16, KVP_F32, KvpError, kvp_abi_version, kvp_check_device_status,
                   kvp_chunk_compress, kvp_eviction_auc, kvp_rank_rows,
                   kvp_compact_kv, kvp_decode_attn, kvp_decode_attn_workspace_size,
                   kvp_future_attn_mass, kvp_future_attn_mass_workspace_size, kvp_future_attn_target,
                   kvp_future_attn_target_workspace_size,
                   kvp_launch_count, kvp_lse_pass,
                   kvp_ring_insert, kvp_select_topk, kvp_soft_topk_budgets, kvp_sparse_lse_pass,
                   kvp_sparse_lse_workspace_size,
                   kvp_topk_cutoffs, load)
from .pipeline import prefill_prune_step

__all__ = [
    "KVP_F32", "KVP_BF16", "KVP_F16", "KvpError", "load", "kvp_lse_pass", "kvp_future_attn_mass",
    "kvp_future_attn_mass_workspace_size", "kvp_future_attn_target",
    "kvp_future_attn_target_workspace_size", "kvp_soft_topk_budgets", "kvp_select_topk",
    "kvp_compact_kv", "kvp_chunk_compress", "kvp_rank_rows", "kvp_eviction_auc", "kvp_ring_insert", "kvp_decode_attn", "kvp_decode_attn_workspace_size",
    "kvp_topk_cutoffs", "kvp_sparse_lse_pass", "kvp_sparse_lse_workspace_size",
    "kvp_check_device_status", "kvp_abi_version", "kvp_launch_count", "prefill_prune_step",
]
