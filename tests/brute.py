"""Brute-force references for tiny inputs, built on library routines.

They materialise the whole S x S attention matrix through scipy's softmax /
logsumexp (a different algorithm from the oracle's streaming per-block
evaluation) and are used only to pin the oracle.
"""
import numpy as np
from scipy.special import logsumexp, softmax


def causal_logits(q, k, scale):
    """[S, S] logits with the causal mask applied as -inf (query rows, key columns)."""
    s = (np.asarray(q, np.float64) @ np.asarray(k, np.float64).T) * scale
    S = s.shape[0]
    return np.where(np.tril(np.ones((S, S), dtype=bool)), s, -np.inf)


def lse(q, k, scale):
    Hq = q.shape[0]
    G = Hq // k.shape[0]
    return np.stack([logsumexp(causal_logits(q[h], k[h // G], scale), axis=1) for h in range(Hq)])


def future_mass(q, k, scale, w):
    Hq, S, _ = q.shape
    Hkv = k.shape[0]
    G = Hq // Hkv
    F = np.zeros((Hkv, S))
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    for h in range(Hq):
        P = softmax(causal_logits(q[h], k[h // G], scale), axis=1)
        F[h // G] += (P * (i >= j + w)).sum(axis=0)
    return F


def decode(q, k, v, scale):
    p = softmax((np.asarray(k, np.float64) @ np.asarray(q, np.float64)) * scale)
    return p @ np.asarray(v, np.float64), p
