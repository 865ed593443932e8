"""Oracle of KVP's budget-agnostic eviction cost of a ranking.

Learning to Evict from Key-Value Cache §1, §3 and §3.1.1: a ranking of a head's cache entries
serves every budget at once (the top-b entries are kept, the rest evicted); its global reward
measures, over all budgets, the future-attention importance of the entries it would evict and
scores the ranking by the area under that cost-versus-budget curve, normalised by the cost of
the optimal ranking.  Readings taken here (the page gives the quantities in words only):

* importance of an entry = its future-attention mass F (the mass pass of this library);
* cost(b) = sum of F over the entries ranked b or later (0-based ranks: budget b keeps ranks
  0 .. b-1), for every budget b = 0 .. T;
* AUC = sum over b = 0 .. T of cost(b) (unit budget steps); the optimal ranking orders entries
  by F, largest first, and the normalised cost is AUC / AUC_optimal (1 for an optimal ranking,
  larger otherwise).
"""
from __future__ import annotations

import numpy as np


def rank_by_scores(scores) -> np.ndarray:
    """0-based ranks: 0 = highest score; ties go to the lower index; NaN ranks last."""
    s = np.asarray(scores, dtype=np.float64)
    T = s.size
    nan = np.isnan(s)
    key = np.where(nan, 0.0, -s) + 0.0
    order = np.lexsort((np.arange(T), key, nan))
    ranks = np.empty(T, dtype=np.int64)
    ranks[order] = np.arange(T)
    return ranks


def eviction_cost_curve(F, ranks) -> np.ndarray:
    """cost[b] = sum of F over entries with rank >= b, b = 0..T."""
    F = np.asarray(F, dtype=np.float64)
    ranks = np.asarray(ranks, dtype=np.int64)
    T = F.size
    by_rank = np.empty(T)
    by_rank[ranks] = F
    return np.array([by_rank[b:].sum() for b in range(T + 1)])


def eviction_auc(F, ranks) -> float:
    return float(eviction_cost_curve(F, ranks).sum())


def optimal_auc(F) -> float:
    return eviction_auc(F, rank_by_scores(F))


def normalized_auc(F, ranks) -> float:
    opt = optimal_auc(F)
    return eviction_auc(F, ranks) / opt if opt > 0 else 1.0
