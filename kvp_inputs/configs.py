"""The five seeded synthetic workloads the hot path is measured and checked on.

Each workload is named by the model it is shaped like and its sizes.  None of
the pages ships data we can use here, so every tensor is synthetic: standard
normal queries/keys/values drawn from a seeded generator, with a few planted
structures (attention-sink keys, retrieval keys) so that the future-attention
mass is not flat.  The recipe itself lives in :mod:`kvp_inputs.gen`.

This module holds sizes only; it contains none of the method's arithmetic.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    name: str
    n_layers: int
    h_q: int
    h_kv: int
    head_dim: int
    seq_len: int            # prefill length S (or cache length T for decode workloads)
    dtype: str              # "f32" | "bf16" | "f16"
    window: int             # protected recent window w of the future-attention target
    n_sink: int
    n_recent: int
    budget: int | None = None            # uniform per-KV-head budget b
    retention: float | None = None       # aggregate retention for learned head-wise budgets
    decode_budgets: tuple = ()           # budgets swept by the decode-eviction workload
    key_scale: tuple | None = None       # per-KV-head key scale ~ U[lo, hi]
    n_sink_keys: int = 0                 # leading tokens whose key is the sink construction
    n_retrieval: int = 0                 # planted retrieval keys per KV head
    seed: int = 0
    kind: str = "prefill"                # "prefill" (F -> select -> compact -> decode) or "decode"
    notes: str = ""

    @property
    def group(self) -> int:
        return self.h_q // self.h_kv

    @property
    def rows(self) -> int:
        """Independent (layer, KV head) rows R."""
        return self.n_layers * self.h_kv

    def scaled(self, **kw) -> "Workload":
        """A smaller copy with the same recipe (for parity runs the oracle finishes in seconds)."""
        return dataclasses.replace(self, **kw)

    def attn_mass_flops(self, seq_len: int | None = None, window: int | None = None) -> float:
        """Algorithmic flops of the row-LSE and future-mass passes: 2*D per scored (query, key)
        pair; the LSE pass scores S(S+1)/2 causal pairs per query head, the mass pass
        (S-w)(S-w+1)/2 masked pairs per query head."""
        S = self.seq_len if seq_len is None else seq_len
        w = self.window if window is None else window
        ww = max(S - w, 0)
        pairs = S * (S + 1) // 2 + ww * (ww + 1) // 2
        return 2.0 * self.head_dim * self.h_q * self.n_layers * pairs


TINY = Workload(
    name="tiny-1L-2q1kv-d64-S256-f32",
    n_layers=1, h_q=2, h_kv=1, head_dim=64, seq_len=256, dtype="f32",
    window=16, n_sink=4, n_recent=16, budget=64,
    n_sink_keys=1, n_retrieval=0, seed=0,
    notes="token 0's key is the group's mean query direction scaled to 3*sqrt(D)",
)

QWEN3_4B_LAYER = Workload(
    name="qwen3-4b-shaped-1L-32q8kv-d128-S8192-bf16",
    n_layers=1, h_q=32, h_kv=8, head_dim=128, seq_len=8192, dtype="bf16",
    window=128, n_sink=4, n_recent=128, budget=2048,
    key_scale=(0.5, 2.0), n_sink_keys=4, n_retrieval=16, seed=1,
)

LLAMA31_8B_32L = Workload(
    name="llama3.1-8b-shaped-32L-32q8kv-d128-S32768-bf16",
    n_layers=32, h_q=32, h_kv=8, head_dim=128, seq_len=32768, dtype="bf16",
    window=64, n_sink=4, n_recent=64, retention=0.15,
    key_scale=(0.5, 2.0), n_sink_keys=4, n_retrieval=16, seed=2,
    notes="per-head budgets from the closed-form Soft-TopK over 256 N(0,1) head scores",
)

QWEN25_15B_DECODE = Workload(
    name="qwen2.5-1.5b-shaped-28L-12q2kv-d128-T120000-f16-decode",
    n_layers=28, h_q=12, h_kv=2, head_dim=128, seq_len=120000, dtype="f16",
    window=0, n_sink=4, n_recent=32, decode_budgets=(512, 1024, 2048, 4096),
    seed=3, kind="decode",
    notes="score = group-summed attention of one decode query over the full cache",
)

QWEN3_8B_131K = Workload(
    name="qwen3-8b-shaped-1L-32q8kv-d128-S131072-bf16",
    n_layers=1, h_q=32, h_kv=8, head_dim=128, seq_len=131072, dtype="bf16",
    window=256, n_sink=4, n_recent=256, budget=16384,
    key_scale=(0.5, 2.0), n_sink_keys=4, n_retrieval=16, seed=4,
)

ALL = (TINY, QWEN3_4B_LAYER, LLAMA31_8B_32L, QWEN25_15B_DECODE, QWEN3_8B_131K)
BY_NAME = {w.name: w for w in ALL}
