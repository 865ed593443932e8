"""Oracle of chunked prefill-compress (one step and the whole loop).

Learning to Evict from Key-Value Cache, §4 and §4.1: long contexts are prefilled in chunks and
the cache is compressed back to the budget after every chunk, with physical tensor compaction;
budgets are uniform across heads and layers; the ranking scores are per token and do not
depend on the query, so a kept token keeps its score.  Each step appends the chunk after the
kept entries (source order is preserved) and applies the selection rule of
:func:`oracle.selection.select_row` (sinks, the most recent tokens, the top-scoring rest) to
the union, then gathers the kept K/V rows, scores and source positions.
"""
from __future__ import annotations

import numpy as np

from .selection import effective_budget, select_row


def chunk_compress_step(cache, n_in: int, chunk_k, chunk_v, chunk_score, pos0: int, budget: int,
                        n_sink: int, n_recent: int):
    """cache: dict of numpy arrays "k", "v" [R, >= n_in, D] (any dtype; copied bytewise),
    "score" [R, >= n_in], "pos" [R, >= n_in] (or None when n_in = 0).  Returns (out, idx, count)
    with out's arrays holding count[r] entries per row (count is the same for every row)."""
    R, C = chunk_score.shape
    T = n_in + C
    b_eff = effective_budget(T, budget, n_sink, n_recent)
    D = chunk_k.shape[2]
    out = {"k": np.zeros((R, b_eff, D), dtype=chunk_k.dtype), "v": np.zeros((R, b_eff, D), dtype=chunk_v.dtype),
           "score": np.zeros((R, b_eff), dtype=np.float32), "pos": np.zeros((R, b_eff), dtype=np.int64)}
    idx = np.full((R, b_eff), -1, dtype=np.int64)
    count = np.zeros(R, dtype=np.int64)
    for r in range(R):
        if n_in:
            uk = np.concatenate([cache["k"][r, :n_in], chunk_k[r]])
            uv = np.concatenate([cache["v"][r, :n_in], chunk_v[r]])
            us = np.concatenate([np.asarray(cache["score"][r, :n_in], np.float32), chunk_score[r]])
            up = np.concatenate([np.asarray(cache["pos"][r, :n_in], np.int64), pos0 + np.arange(C)])
        else:
            uk, uv, us, up = chunk_k[r], chunk_v[r], np.asarray(chunk_score[r], np.float32), pos0 + np.arange(C)
        keep = select_row(us.astype(np.float64), budget, n_sink, n_recent)
        n = keep.size
        idx[r, :n] = keep
        count[r] = n
        out["k"][r, :n] = uk[keep]
        out["v"][r, :n] = uv[keep]
        out["score"][r, :n] = us[keep]
        out["pos"][r, :n] = up[keep]
    return out, idx, count


def chunked_prefill_compress(k, v, scores, chunk_len: int, budget: int, n_sink: int, n_recent: int):
    """Whole loop over a sequence k, v [R, S, D], scores [R, S] in chunks of chunk_len.
    Returns the final cache dict (count entries per row) and the per-step counts."""
    R, S = scores.shape
    cache, n = None, 0
    counts = []
    for p0 in range(0, S, chunk_len):
        p1 = min(S, p0 + chunk_len)
        cache, _, cnt = chunk_compress_step(cache, n, k[:, p0:p1], v[:, p0:p1], scores[:, p0:p1], p0,
                                            budget, n_sink, n_recent)
        n = int(cnt[0])
        counts.append(n)
    return cache, counts
