"""Pins of the eviction-cost AUC oracle: the closed form sum_t (rank_t + 1) F_t (summing the
cost curve by entries instead of budgets), the optimum against brute force over every ranking of
tiny rows, the rearrangement bound for random rankings, the shape of the cost curve, and the
score ranking against numpy's stable argsort (the selection rule's tie and NaN order)."""
import itertools

import numpy as np
import pytest

from oracle.auc import eviction_auc, eviction_cost_curve, normalized_auc, optimal_auc, rank_by_scores
from oracle.selection import select_row


@pytest.mark.parametrize("seed", range(6))
def test_closed_form_and_curve(seed):
    rng = np.random.default_rng(seed)
    T = int(rng.integers(1, 300))
    F = rng.exponential(size=T) * (rng.random(T) < 0.8)
    ranks = rng.permutation(T)
    curve = eviction_cost_curve(F, ranks)
    assert abs(curve[0] - F.sum()) < 1e-9 and curve[-1] == 0.0
    assert (np.diff(curve) <= 1e-12).all()
    assert abs(eviction_auc(F, ranks) - ((ranks + 1) * F).sum()) < 1e-8 * max(1.0, F.sum() * T)


@pytest.mark.parametrize("T", [1, 2, 3, 5, 6])
def test_optimum_is_the_best_of_all_rankings(T):
    rng = np.random.default_rng(T)
    F = np.round(rng.exponential(size=T), 1)          # ties included
    best = min(eviction_auc(F, np.array(p)) for p in itertools.permutations(range(T)))
    assert abs(optimal_auc(F) - best) < 1e-12


def test_random_rankings_cost_at_least_the_optimum():
    rng = np.random.default_rng(11)
    F = rng.exponential(size=500)
    opt = optimal_auc(F)
    for _ in range(20):
        assert normalized_auc(F, rng.permutation(500)) >= 1.0
    assert abs(normalized_auc(F, rank_by_scores(F)) - 1.0) < 1e-15
    assert opt > 0


def test_score_ranking_matches_stable_argsort_and_the_selection_rule():
    rng = np.random.default_rng(5)
    s = np.round(rng.standard_normal(400), 1)
    want = np.empty(400, dtype=np.int64)
    want[np.argsort(-s, kind="stable")] = np.arange(400)
    assert (rank_by_scores(s) == want).all()
    s2 = s.copy()
    s2[[3, 50]] = np.nan
    r2 = rank_by_scores(s2)
    assert set(r2[[3, 50]].tolist()) == {398, 399} and r2[3] < r2[50]
    # the top-b of the ranking is what the selection keeps without sinks or window
    for b in (1, 17, 200, 399):
        assert (np.flatnonzero(rank_by_scores(s) < b) == select_row(s, b, 0, 0)).all()
