"""fp64/integer oracle for budgeted per-KV-head selection and K/V compaction.

Selection (KVpop, "The KVpop Scoring Module" and Figure 1; Learning to Evict
from Key-Value Cache, §1 and §A.2; How much KV cache can you prune, "What we
did"): a row of T cached tokens keeps the first ``n_sink`` tokens, the newest
``n_recent`` tokens, and fills the rest of the budget b with the highest-scored
remaining tokens; the budget counts the sinks and the recent window (the
KVpop worked example keeps 2 + 3 + 4 = 9 = B tokens).

Readings where the pages are silent:

* ties go to the lower token index; -0.0 equals +0.0; NaN ranks below -inf;
* T <= b keeps all T tokens; b < n_sink + n_recent is raised to
  n_sink + n_recent; the kept count is then exactly the effective budget;
* kept indices are listed in ascending token order.

The top-k is a full sort with the comparator (score descending, index
ascending) -- the textbook definition a radix select reaches faster.

Compaction (Learning to Evict, §4.1 "physical tensor compaction"; How much
KV cache can you prune, "Conclusion": the kept entries are copied into a new
tensor): row m of the compacted cache is row idx[m] of the source, byte for byte.
"""
from __future__ import annotations

import numpy as np


def effective_budget(T: int, b: int, n_sink: int, n_recent: int) -> int:
    if b < 0:
        raise ValueError("negative budget")
    if T <= b:
        return T
    return min(T, max(b, n_sink + n_recent))


def select_row(scores, b: int, n_sink: int, n_recent: int) -> np.ndarray:
    """Kept token indices (ascending) of one row of scores."""
    s = np.asarray(scores, dtype=np.float64)
    T = s.size
    b_eff = effective_budget(T, b, n_sink, n_recent)
    if b_eff >= T:
        return np.arange(T, dtype=np.int64)
    sinks = np.arange(n_sink)
    recent = np.arange(T - n_recent, T)
    middle = np.arange(n_sink, T - n_recent)
    k = b_eff - n_sink - n_recent
    sm = s[middle]
    nan = np.isnan(sm)
    desc = np.where(nan, 0.0, -sm) + 0.0          # + 0.0 turns -0.0 into +0.0
    order = np.lexsort((middle, desc, nan))       # primary: non-NaN first, then score desc, then index asc
    chosen = middle[order[:k]]
    return np.sort(np.concatenate([sinks, chosen, recent])).astype(np.int64)


def select_topk(scores, budgets, n_sink: int, n_recent: int, b_max: int | None = None):
    """Rows of ``scores`` [R, T] -> (idx [R, b_max] ascending, -1 padded; count [R])."""
    s = np.asarray(scores)
    R, T = s.shape
    budgets = np.broadcast_to(np.asarray(budgets, dtype=np.int64), (R,))
    kept = [select_row(s[r], int(budgets[r]), n_sink, n_recent) for r in range(R)]
    width = max((x.size for x in kept), default=0) if b_max is None else int(b_max)
    idx = np.full((R, width), -1, dtype=np.int64)
    count = np.zeros(R, dtype=np.int64)
    for r, x in enumerate(kept):
        idx[r, :x.size] = x
        count[r] = x.size
    return idx, count


def compact_kv(k, v, idx, count):
    """k, v [R, T, D] -> kc, vc [R, width, D] with row m = source row idx[r, m] for m < count[r];
    rows m >= count[r] are zero."""
    k = np.asarray(k)
    v = np.asarray(v)
    R, T, D = k.shape
    width = idx.shape[1]
    kc = np.zeros((R, width, D), dtype=k.dtype)
    vc = np.zeros((R, width, D), dtype=v.dtype)
    for r in range(R):
        n = int(count[r])
        kc[r, :n] = k[r, idx[r, :n]]
        vc[r, :n] = v[r, idx[r, :n]]
    return kc, vc
