"""fp64 / integer oracle of the static (ring) decode cache with in-place eviction.

How much KV cache can you prune before quality degrades, "What we did" (the
attention-score policy keeps the first four tokens, always keeps the newest
32 and fills the remaining space with the older tokens that received the most
attention) and "Conclusion" (a ring or static cache reserves a fixed region and
overwrites old entries in place instead of selecting and copying).

One decode step on one row of a cache with ``cap`` slots, after the step's
attention has been added to the slots' cumulative scores:

* while the cache is not full the new token is appended at slot ``fill``;
* otherwise the evictable slots are those whose token position p satisfies
  n_sink <= p <= new_pos - n_recent (not a sink, not among the n_recent newest
  tokens counting the new one); the slot with the lowest score is overwritten,
  ties going to the slot holding the NEWER token (the mirror of the selection
  rule that keeps the lower index among equal scores); NaN scores are evicted
  first;
* the new token's slot gets position new_pos and score 0.
"""
from __future__ import annotations

import numpy as np


def ring_victim(pos, score, fill: int, cap: int, new_pos: int, n_sink: int, n_recent: int) -> int:
    """Slot that receives the new token (-1 if the cache is full and nothing is evictable)."""
    if fill < cap:
        return fill
    pos = np.asarray(pos)
    score = np.asarray(score, dtype=np.float64)
    best, best_key = -1, None
    for m in range(cap):
        p = int(pos[m])
        if p < n_sink or p > new_pos - n_recent:
            continue
        s = score[m]
        # smallest score first (NaN below everything, -0.0 == +0.0), then the newest token
        key = (0, 0.0, -p) if np.isnan(s) else (1, s + 0.0, -p)
        if best_key is None or key < best_key:
            best, best_key = m, key
    return best


def ring_insert(kc, vc, pos, score, fill, new_k, new_v, new_pos: int, n_sink: int, n_recent: int):
    """Apply one insertion to every row in place: kc, vc [R, cap, D]; pos int [R, cap];
    score [R, cap]; fill int [R]; new_k, new_v [R, D].  Returns the chosen slots [R]."""
    R, cap, _ = kc.shape
    slots = np.full(R, -1, dtype=np.int64)
    for r in range(R):
        m = ring_victim(pos[r], score[r], int(fill[r]), cap, new_pos, n_sink, n_recent)
        slots[r] = m
        if m < 0:
            continue
        kc[r, m] = new_k[r]
        vc[r, m] = new_v[r]
        pos[r, m] = new_pos
        score[r, m] = 0.0
        if fill[r] < cap:
            fill[r] += 1
    return slots
