"""Seeded synthetic workloads (sizes + generators).  Holds none of the method's arithmetic;
shared by the CUDA path's tests and benchmark and by the oracle's tests."""
from .configs import (ALL, BY_NAME, LLAMA31_8B_32L, QWEN3_4B_LAYER, QWEN3_8B_131K,
                      QWEN25_15B_DECODE, TINY, Workload)
from .gen import (make_decode_cache, make_head_scores, make_prefill, make_prefill_layer,
                  make_scores, make_static_ranks, torch_dtype)

__all__ = [
    "ALL", "BY_NAME", "TINY", "QWEN3_4B_LAYER", "LLAMA31_8B_32L", "QWEN25_15B_DECODE",
    "QWEN3_8B_131K", "Workload", "make_prefill", "make_prefill_layer", "make_decode_cache",
    "make_head_scores", "make_scores", "make_static_ranks", "torch_dtype",
]
