"""fp64 / integer oracle of KVpop's running top-k cutoff and the sparse attention normaliser.

Followed passages (KVpop -- Key-Value Cache Compression with Predictive Online Pruning):

* "Efficient Online Pruning" and "Fenwick-tree cut-off computation (Algorithm 2)": every
  token of a KV head carries a static rank (a permutation; smaller rank = more important).
  At query position q the token t = q - w leaves the protected window; if it is not one of
  the first s (sink) tokens its rank is inserted into a Fenwick tree over the ranks.  Once at
  least k tokens are eligible, the cutoff tau_q is the rank of the k-th best eligible token,
  found by binary lifting on the tree's prefix counts; before that tau_q = -1.
* The sparse attention of query q covers the sinks, the protected window (q - w, q] and the
  eligible tokens of rank <= tau_q ("attends to the union of sink tokens, the protected
  window, and the top-k eligible tokens").  While fewer than k tokens are eligible (tau_q = -1)
  the top-k eligible set is all of them (the plainest reading of "top-k" with fewer than k
  candidates; the pages give no rule for it).
* "Delayed Memory Scoring": the future-attention target may reuse the sparse log-normalisers
  of this attention; :func:`sparse_row_lse` is that normaliser, ln of the summed exponentiated
  logits over the kept keys.

Ranks here are 0-based (the page's worked example numbers them from 1).
"""
from __future__ import annotations

import numpy as np

from .attention_mass import _as_f64


class Fenwick:
    """Fenwick (binary indexed) tree of counts over positions 1..n."""

    def __init__(self, n: int):
        self.n = int(n)
        self.tree = [0] * (self.n + 1)

    def add(self, i: int, v: int = 1) -> None:
        """counts[i] += v (1-based i)."""
        while i <= self.n:
            self.tree[i] += v
            i += i & -i

    def prefix(self, i: int) -> int:
        """counts[1] + ... + counts[i]."""
        s = 0
        while i > 0:
            s += self.tree[i]
            i -= i & -i
        return s

    def find_by_prefix_count(self, k: int) -> int:
        """Smallest i with prefix(i) >= k (k >= 1), by binary lifting; n + 1 if none."""
        pos, rem = 0, int(k)
        step = 1
        while step * 2 <= self.n:
            step *= 2
        while step:
            nxt = pos + step
            if nxt <= self.n and self.tree[nxt] < rem:
                pos = nxt
                rem -= self.tree[nxt]
            step //= 2
        return pos + 1


def fenwick_cutoffs(ranks, n_sink: int, window: int, k: int) -> np.ndarray:
    """tau[q] for q = 0..S-1 of one KV head (Algorithm 2); ranks: a permutation of 0..S-1."""
    ranks = np.asarray(ranks, dtype=np.int64)
    S = ranks.size
    if k < 1:
        raise ValueError("k must be >= 1")
    tree = Fenwick(S)
    tau = np.full(S, -1, dtype=np.int64)
    eligible = 0
    for q in range(S):
        t = q - window
        if t >= n_sink:
            tree.add(int(ranks[t]) + 1)
            eligible += 1
        if eligible >= k:
            tau[q] = tree.find_by_prefix_count(k) - 1
    return tau


def sparse_keep(q: int, j: int, rank_j: int, tau_q: int, n_sink: int, window: int) -> bool:
    """Whether query q attends to key j under the running top-k mask."""
    if j > q:
        return False
    if j < n_sink or j > q - window:
        return True
    return tau_q < 0 or rank_j <= tau_q


def sparse_mask(ranks, tau, n_sink: int, window: int) -> np.ndarray:
    """Boolean [S, S] mask (query, key) of one KV head."""
    ranks = np.asarray(ranks, dtype=np.int64)
    tau = np.asarray(tau, dtype=np.int64)
    S = ranks.size
    qq = np.arange(S)[:, None]
    jj = np.arange(S)[None, :]
    causal = jj <= qq
    protected = (jj < n_sink) | (jj > qq - window)
    top = (tau[:, None] < 0) | (ranks[None, :] <= tau[:, None])
    return causal & (protected | top)


def sparse_row_lse(q, k, ranks, tau, scale: float, n_sink: int, window: int, rows=None) -> np.ndarray:
    """lse[h_q, i] = ln sum_{j kept for (h_q // G, i)} exp(scale * q[h_q, i] . k[h_q // G, j]).

    q: [H_q, S, D]; k: [H_kv, S, D]; ranks, tau: [H_kv, S].  ``rows`` optionally lists the query
    positions to evaluate (the result then has shape [H_q, len(rows)])."""
    q = _as_f64(q)
    k = _as_f64(k)
    ranks = np.asarray(ranks, dtype=np.int64)
    tau = np.asarray(tau, dtype=np.int64)
    Hq, S, _ = q.shape
    Hkv = k.shape[0]
    G = Hq // Hkv
    rows = np.arange(S) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.empty((Hq, rows.size))
    jj = np.arange(S)[None, :]
    blk = max(1, (1 << 22) // max(S, 1))
    for h in range(Hkv):
        for b0 in range(0, rows.size, blk):
            ii = rows[b0:b0 + blk][:, None]
            t = tau[h][ii]
            keep = (jj <= ii) & ((jj < n_sink) | (jj > ii - window) | (t < 0) | (ranks[h][None, :] <= t))
            for g in range(G):
                s = (q[h * G + g, ii[:, 0]] @ k[h].T) * scale
                s = np.where(keep, s, -np.inf)
                m = s.max(axis=1, keepdims=True)
                out[h * G + g, b0:b0 + blk] = m[:, 0] + np.log(np.exp(s - m).sum(axis=1))
    return out
