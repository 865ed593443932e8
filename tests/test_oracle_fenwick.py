"""Pins of the running top-k cutoff (KVpop, Algorithm 2) and of the sparse log-normaliser.

* the page's worked Fenwick example (tests/golden/kvpop_fenwick_example.json);
* brute force: tau_q is the k-th smallest rank among the tokens s..q-w, found here by a
  sort of that slice, on many small random permutations and budgets;
* invariants: tau is non-increasing once defined, exactly k eligible tokens have rank <= tau_q;
* the sparse LSE against a logsumexp over a mask built per query by sorting, against the dense
  causal LSE when every eligible token is kept, and against ln(kept count) for uniform
  attention (closed form)."""
import json
import os

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle
from oracle.fenwick import Fenwick, fenwick_cutoffs, sparse_mask, sparse_row_lse

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kvpop_fenwick_example.json")


def test_page_worked_example():
    ex = json.load(open(GOLDEN))
    tree = Fenwick(ex["n"])
    for i, r in enumerate(ex["inserts_1based"]):
        tree.add(r)
        counts = [tree.prefix(j + 1) - tree.prefix(j) for j in range(ex["n"])]
        assert counts == ex["counts_after_each_insert"][i]
        want = ex["tau_1based_after_each_insert"][i]
        if want is not None:
            assert tree.find_by_prefix_count(ex["k"]) == want
    assert tree.prefix(4) == ex["prefix_count_at_rank4_after_third"]
    # the same stream through the cutoff routine (s = 0, w = 0: token t is eligible at q = t)
    ranks0 = [r - 1 for r in ex["inserts_1based"]]
    tau = fenwick_cutoffs(ranks0, n_sink=0, window=0, k=ex["k"])
    assert tau.tolist() == [-1, 2, 2]


def brute_cutoffs(ranks, s, w, k):
    S = len(ranks)
    out = np.full(S, -1)
    for q in range(S):
        elig = ranks[s:max(s, q - w + 1)]
        if len(elig) >= k:
            out[q] = np.sort(elig)[k - 1]
    return out


@pytest.mark.parametrize("seed", range(12))
def test_cutoffs_match_brute_force(seed):
    rng = np.random.default_rng(seed)
    S = int(rng.integers(1, 200))
    ranks = rng.permutation(S)
    for s, w, k in [(0, 0, 1), (4, 16, 8), (int(rng.integers(0, 10)), int(rng.integers(0, 40)),
                                             int(rng.integers(1, 60))), (0, S + 3, 2), (2, 1, S + 1)]:
        got = fenwick_cutoffs(ranks, s, w, k)
        want = brute_cutoffs(ranks, s, w, k)
        assert (got == want).all(), (S, s, w, k)
        defined = got >= 0
        if defined.any():
            first = int(np.argmax(defined))
            assert defined[first:].all()
            assert (np.diff(got[first:]) <= 0).all()
            for q in np.flatnonzero(defined)[:: max(1, S // 17)]:
                elig = ranks[s:q - w + 1]
                assert int((elig <= got[q]).sum()) == k


def test_fenwick_binary_lifting_against_linear_scan():
    rng = np.random.default_rng(7)
    for n in (1, 2, 3, 8, 13, 64, 100):
        tree = Fenwick(n)
        counts = np.zeros(n + 1, dtype=int)
        for _ in range(3 * n):
            i = int(rng.integers(1, n + 1))
            tree.add(i)
            counts[i] += 1
            cum = np.cumsum(counts)
            for k in range(1, int(cum[-1]) + 1, max(1, int(cum[-1]) // 5)):
                assert tree.find_by_prefix_count(k) == int(np.argmax(cum >= k))


def _rand_qk(rng, Hq, Hkv, S, D):
    return rng.standard_normal((Hq, S, D)), rng.standard_normal((Hkv, S, D))


def test_sparse_lse_against_per_query_sort():
    rng = np.random.default_rng(3)
    Hq, Hkv, S, D, s, w, k = 4, 2, 90, 16, 3, 7, 10
    q, kk = _rand_qk(rng, Hq, Hkv, S, D)
    ranks = np.stack([rng.permutation(S) for _ in range(Hkv)])
    tau = np.stack([fenwick_cutoffs(ranks[h], s, w, k) for h in range(Hkv)])
    got = sparse_row_lse(q, kk, ranks, tau, 0.25, s, w)
    G = Hq // Hkv
    for hq in range(Hq):
        h = hq // G
        for i in range(S):
            elig = np.arange(s, max(s, i - w + 1))
            top = elig[np.argsort(ranks[h][elig], kind="stable")[:k]]
            keep = sorted(set(range(min(s, i + 1))) | set(range(max(0, i - w + 1), i + 1)) | set(top.tolist()))
            want = logsumexp(0.25 * (kk[h][keep] @ q[hq, i]))
            assert abs(got[hq, i] - want) < 1e-12
    mask = sparse_mask(ranks[0], tau[0], s, w)
    assert mask.sum(axis=1).max() <= s + w + k


def test_sparse_lse_keeping_everything_is_dense():
    rng = np.random.default_rng(4)
    Hq, Hkv, S, D = 2, 1, 70, 8
    q, kk = _rand_qk(rng, Hq, Hkv, S, D)
    ranks = rng.permutation(S)[None]
    tau = fenwick_cutoffs(ranks[0], 2, 5, S + 1)[None]          # never k eligible: tau = -1
    assert (tau == -1).all()
    dense = oracle.row_lse(q, kk, 0.3)
    assert np.allclose(sparse_row_lse(q, kk, ranks, tau, 0.3, 2, 5), dense, atol=1e-12)


def test_sparse_lse_uniform_attention_closed_form():
    S, s, w, k = 120, 4, 16, 9
    q = np.zeros((2, S, 8))
    kk = np.random.default_rng(5).standard_normal((1, S, 8))
    ranks = np.random.default_rng(6).permutation(S)[None]
    tau = fenwick_cutoffs(ranks[0], s, w, k)[None]
    got = sparse_row_lse(q, kk, ranks, tau, 1.0, s, w)
    i = np.arange(S)
    elig = np.maximum(0, i - w - s + 1)
    kept = np.minimum(w, i + 1) + np.minimum(s, np.maximum(0, i - w + 1)) + np.minimum(k, elig)
    assert np.allclose(got, np.log(kept)[None], atol=1e-12)
