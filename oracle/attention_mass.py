"""fp64 oracle for the causal row log-sum-exp and the future-attention mass.

Definitions followed (KVpop — Key-Value Cache Compression with Predictive
Online Pruning):

* "Delayed Memory Scoring", the worked LSE example: the log-normaliser of
  query d is the log of the summed exponentiated logits over the keys the
  causal mask lets it see (keys t' <= d, the diagonal included).
* "Defining Future Attention Utility" and Figure 2: the future-attention mass
  of key t is the softmax probability it receives from every query d that
  has left the protected window, d >= t + w (the worked example's count
  N_t = S - (t + w) fixes the boundary as inclusive); the transposed pass
  obtains it as exp(logit - LSE(d)) summed over those queries.
* Heads: the GQA group of KV head h is query heads h*G ... h*G+G-1, and the
  mass is summed over the group (raw sum, no count normalisation, no log).
* Logits are q.k * scale with scale = 1/sqrt(D) (the standard reading of the
  garbled kernel in "Background: Linear Attention").

Everything is computed in float64 from the exact (already rounded) inputs.
The matrix product is a library step (numpy matmul); masking, max, exp, log
and sums are written out.  Blocks only bound memory; they do not change what
is summed.
"""
from __future__ import annotations

import numpy as np

_BLOCK_ELEMS = 1 << 23  # elements of one fp64 logit block (64 MiB)


def _as_f64(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def row_lse(q, k, scale: float, rows=None) -> np.ndarray:
    """lse[h_q, i] = ln sum_{j <= i} exp(scale * q[h_q, i] . k[h_q // G, j]).

    q: [H_q, S, D]; k: [H_kv, S, D].  ``rows`` optionally lists the query
    positions to evaluate (the result then has shape [H_q, len(rows)]).
    """
    q = _as_f64(q)
    k = _as_f64(k)
    Hq, S, D = q.shape
    Hkv = k.shape[0]
    G = Hq // Hkv
    rows = np.arange(S) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.empty((Hq, rows.size))
    order = np.argsort(rows, kind="stable")
    blk = max(1, _BLOCK_ELEMS // max(S, 1))
    for h in range(Hq):
        kh = k[h // G]
        for b0 in range(0, rows.size, blk):
            sel = order[b0:b0 + blk]
            ii = rows[sel]
            jmax = int(ii.max()) + 1
            s = (q[h, ii] @ kh[:jmax].T) * scale
            visible = np.arange(jmax)[None, :] <= ii[:, None]
            s = np.where(visible, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            out[h, sel] = m[:, 0] + np.log(np.exp(s - m).sum(axis=1))
    return out


def future_attn_mass(q, k, lse, scale: float, window: int, keys=None) -> np.ndarray:
    """F[h_kv, j] = sum_{g < G} sum_{i = j + w}^{S-1} exp(scale * q[h_kv*G+g, i] . k[h_kv, j] - lse[h_kv*G+g, i]).

    ``lse`` must be this oracle's own [H_q, S] row LSE.  ``keys`` optionally
    lists key positions (result [H_kv, len(keys)]); by default every key.
    Keys with j > S-1-w receive no query and get exactly 0.
    """
    q = _as_f64(q)
    k = _as_f64(k)
    lse = _as_f64(lse)
    Hq, S, D = q.shape
    Hkv = k.shape[0]
    G = Hq // Hkv
    keys = np.arange(S) if keys is None else np.asarray(keys, dtype=np.int64)
    F = np.zeros((Hkv, keys.size))
    kblk = 256
    for h in range(Hkv):
        for a in range(0, keys.size, kblk):
            jj = keys[a:a + kblk]
            first = int(jj.min()) + window          # first query any key of this block can receive
            if first > S - 1:
                continue
            qblk = max(1, _BLOCK_ELEMS // jj.size)
            kj = k[h, jj]
            acc = np.zeros(jj.size)
            for g in range(G):
                hq = h * G + g
                for i0 in range(first, S, qblk):
                    ii = np.arange(i0, min(S, i0 + qblk))
                    s = (q[hq, ii] @ kj.T) * scale
                    p = np.exp(s - lse[hq, ii][:, None])
                    after_window = ii[:, None] >= jj[None, :] + window
                    acc += np.where(after_window, p, 0.0).sum(axis=0)
            F[h, a:a + jj.size] = acc
    return F


def future_attn_mass_per_head(q, k, lse, scale: float, window: int) -> np.ndarray:
    """F_g[h_q, j] = sum_{i = j + w}^{S-1} exp(scale * q[h_q, i] . k[h_q // G, j] - lse[h_q, i]):
    the future-attention mass of every key from each query head separately (KVpop, "Defining
    Future Attention Utility": the mass is formed per query head g before the group
    aggregation)."""
    q = _as_f64(q)
    k = _as_f64(k)
    lse = _as_f64(lse)
    Hq, S, _ = q.shape
    G = Hq // k.shape[0]
    out = np.zeros((Hq, S))
    for hq in range(Hq):
        out[hq] = future_attn_mass(q[hq:hq + 1], k[hq // G:hq // G + 1], lse[hq:hq + 1], scale, window)[0]
    return out


def kvpop_target(F_heads, window: int, group: int, eps: float = 0.0, aggregate: str = "max_log"):
    """KVpop's supervision target from per-query-head future mass (KVpop, "Defining Future
    Attention Utility", worked example, and "Alternative Aggregation Methods"):

        N_t = max(1, S - (t + w))                 count normalisation
        m_g(t) = F_g(t) / N_t                      mean future attention of query head g
        max_log:   r(h, t) = max_g log(eps + m_g(t))
        mean_prob: r(h, t) = log(eps + (1/G) sum_g m_g(t))   (the probability-space mean)

    F_heads: [H_q, S] -> r: [H_q // G, S]."""
    F = np.asarray(F_heads, dtype=np.float64)
    Hq, S = F.shape
    t = np.arange(S)
    N = np.maximum(1, S - (t + window)).astype(np.float64)
    m = F / N[None, :]
    m = m.reshape(Hq // group, group, S)
    with np.errstate(divide="ignore"):
        if aggregate == "max_log":
            return np.log(eps + m).max(axis=1)
        if aggregate == "mean_prob":
            return np.log(eps + m.mean(axis=1))
    raise ValueError(aggregate)
