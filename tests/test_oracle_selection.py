"""Pins of the selection / compaction oracle (no GPU): the KVpop worked budget
example, exhaustive brute force on tiny rows, and the invariants the pages
state (sinks and window always kept, budget met exactly, nested subsets)."""
import itertools
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_kvpop_worked_budget_example():
    ex = json.load(open(os.path.join(GOLDEN, "kvpop_budget_example.json")))
    kept = oracle.select_row(np.array(ex["scores"]), ex["budget"], ex["n_sink"], ex["n_recent"])
    assert kept.tolist() == ex["kept"]
    assert kept.size == ex["budget"] == ex["n_sink"] + ex["n_recent"] + 4


def _brute_kept(s, b, n_sink, n_recent):
    """Among all subsets of the middle with the needed size, the kept ones maximise the
    (exact, integer) score sum; ties go to the lexicographically smallest index tuple."""
    T = s.size
    b_eff = min(T, max(b, n_sink + n_recent)) if T > b else T
    if b_eff >= T:
        return list(range(T))
    middle = range(n_sink, T - n_recent)
    k = b_eff - n_sink - n_recent
    best = None
    for c in itertools.combinations(middle, k):
        key = (sum(int(s[i]) for i in c), [-i for i in c])
        if best is None or key > best[0]:
            best = (key, c)
    return sorted(list(range(n_sink)) + list(best[1]) + list(range(T - n_recent, T)))


@pytest.mark.parametrize("seed", range(12))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(seed)
    T = int(rng.integers(4, 13))
    s = rng.integers(-3, 4, size=T).astype(np.float64)   # heavy ties
    n_sink = int(rng.integers(0, 3))
    n_recent = int(rng.integers(0, 3))
    for b in range(0, T + 2):
        got = oracle.select_row(s, b, n_sink, n_recent).tolist()
        assert got == _brute_kept(s, b, n_sink, n_recent), (s, b, n_sink, n_recent)


def _check_invariants(s, b, n_sink, n_recent, kept):
    T = s.size
    b_eff = oracle.effective_budget(T, b, n_sink, n_recent)
    assert kept.size == b_eff
    assert (np.diff(kept) > 0).all()
    if b_eff < T:
        assert set(range(n_sink)) <= set(kept.tolist())
        assert set(range(T - n_recent, T)) <= set(kept.tolist())
        ks = set(kept.tolist())
        mid = [i for i in range(n_sink, T - n_recent)]
        kept_mid = [i for i in mid if i in ks]
        drop_mid = [i for i in mid if i not in ks]
        if kept_mid and drop_mid:
            def key(i):
                v = s[i]
                return (0, 0.0, i) if np.isnan(v) else (1, v + 0.0, -i)
            assert min(key(i) for i in kept_mid) > max(key(i) for i in drop_mid)


@pytest.mark.parametrize("T,n_sink,n_recent", [(300, 4, 16), (64, 0, 0), (50, 4, 46), (20, 8, 8)])
def test_invariants_random(T, n_sink, n_recent):
    rng = np.random.default_rng(T)
    s = np.round(rng.standard_normal(T) * 4) / 4
    for b in (0, 1, n_sink + n_recent, n_sink + n_recent + 1, T // 2, T - 1, T, T + 5):
        _check_invariants(s, b, n_sink, n_recent, oracle.select_row(s, b, n_sink, n_recent))


def test_nested_across_budgets():
    """Learning to Evict, §3 / §A.1: with a strict ranking the optimal subsets are nested,
    so eviction at any budget is a prefix of one ranking."""
    rng = np.random.default_rng(1)
    s = np.round(rng.standard_normal(200) * 3) / 3
    prev = set()
    for b in range(20, 201, 7):
        cur = set(oracle.select_row(s, b, 4, 16).tolist())
        assert prev <= cur
        prev = cur


def test_zero_fill_is_sinks_plus_window():
    """k = 0 (b = n_sink + n_recent) keeps exactly the sinks and the recent window
    (the sinks-plus-recent policy of How much KV cache can you prune)."""
    s = np.arange(100, dtype=np.float64)[::-1].copy()
    kept = oracle.select_row(s, 36, 4, 32)
    assert kept.tolist() == list(range(4)) + list(range(68, 100))


def test_signed_zero_nan_inf():
    s = np.array([9, 9, -0.0, np.nan, 0.0, -np.inf, np.inf, np.nan, 1.0, -1.0, 9, 9], dtype=np.float64)
    # middle = indices 2..9; order: inf(6), 1.0(8), -0.0(2) == 0.0(4) -> 2 first, -1.0(9), -inf(5), nan(3), nan(7)
    want_order = [6, 8, 2, 4, 9, 5, 3, 7]
    for k in range(0, 9):
        kept = oracle.select_row(s, 4 + k, 2, 2)
        assert kept.tolist() == sorted([0, 1, 10, 11] + want_order[:k])


def test_select_topk_padding_and_counts():
    rng = np.random.default_rng(3)
    s = rng.standard_normal((3, 40))
    idx, count = oracle.select_topk(s, [10, 45, 2], 2, 3, b_max=48)
    assert count.tolist() == [10, 40, 5]
    assert (idx[0, 10:] == -1).all() and (idx[1, :40] == np.arange(40)).all()
    assert idx[2, :5].tolist() == [0, 1, 37, 38, 39]


def test_compact_gathers_rows_bytewise():
    rng = np.random.default_rng(4)
    k = rng.integers(0, 2 ** 16, size=(2, 30, 8)).astype(np.uint16)
    v = rng.integers(0, 2 ** 16, size=(2, 30, 8)).astype(np.uint16)
    idx, count = oracle.select_topk(rng.standard_normal((2, 30)), [7, 12], 1, 2, b_max=16)
    kc, vc = oracle.compact_kv(k, v, idx, count)
    for r in range(2):
        for m in range(int(count[r])):
            assert kc[r, m].tobytes() == k[r, idx[r, m]].tobytes()
            assert vc[r, m].tobytes() == v[r, idx[r, m]].tobytes()
        assert not kc[r, int(count[r]):].any()
