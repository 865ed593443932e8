"""Pins of the KVpop target oracle (no GPU): the page's worked example, brute force of the
per-head mass, and the properties of the count normalisation."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from tests import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_kvpop_worked_target_example():
    ex = json.load(open(os.path.join(GOLDEN, "kvpop_target_example.json")))
    S, t, w, G = ex["S"], ex["t"], ex["window"], ex["group"]
    F_heads = np.zeros((G, S))
    for g in range(G):
        F_heads[g, t] = sum(ex["future_probs"][f"g{g}"])
    r = oracle.kvpop_target(F_heads, w, G, eps=0.0)
    assert max(1, S - (t + w)) == ex["N_t"]
    np.testing.assert_allclose(F_heads[:, t] / ex["N_t"], ex["means"], atol=1e-15)
    np.testing.assert_allclose(np.log(ex["means"]), ex["logs"], atol=ex["print_tolerance"])
    assert abs(r[0, t] - ex["target"]) < ex["print_tolerance"]
    # probability-space mean of the same example: log((0.25 + 0.10) / 2)
    rm = oracle.kvpop_target(F_heads, w, G, eps=0.0, aggregate="mean_prob")
    assert abs(rm[0, t] - math.log(0.175)) < 1e-12


@pytest.mark.parametrize("Hq,Hkv,S,w", [(4, 2, 30, 3), (3, 1, 25, 0), (2, 2, 17, 16)])
def test_per_head_mass_matches_brute_force(Hq, Hkv, S, w):
    rng = np.random.default_rng(S + w)
    q = rng.standard_normal((Hq, S, 8))
    k = rng.standard_normal((Hkv, S, 8))
    lse = oracle.row_lse(q, k, 0.4)
    Fh = oracle.future_attn_mass_per_head(q, k, lse, 0.4, w)
    G = Hq // Hkv
    for hq in range(Hq):
        want = brute.future_mass(q[hq:hq + 1], k[hq // G:hq // G + 1], 0.4, w)[0]
        np.testing.assert_allclose(Fh[hq], want, rtol=1e-12, atol=1e-14)
    # the group sum of the per-head mass is the raw future mass
    np.testing.assert_allclose(Fh.reshape(Hkv, G, S).sum(1), oracle.future_attn_mass(q, k, lse, 0.4, w),
                               rtol=1e-12, atol=1e-14)


def test_uniform_attention_target_closed_form():
    """q.k = 0: p_ij = 1/(i+1), so m(t) = (H_S - H_{t+w}) / (S - t - w) for every head and the
    max over identical heads equals each head's log mean."""
    S, w, G = 40, 5, 3
    Fh = np.zeros((G, S))
    H = np.concatenate([[0.0], np.cumsum(1.0 / np.arange(1, S + 1))])
    for t in range(S):
        if t + w <= S - 1:
            Fh[:, t] = H[S] - H[t + w]
    r = oracle.kvpop_target(Fh, w, G, eps=1e-30)
    for t in range(S - w):
        assert abs(r[0, t] - math.log((H[S] - H[t + w]) / (S - t - w))) < 1e-12
    # keys without future queries: N_t = 1, F = 0 -> log(eps)
    assert np.allclose(r[0, S - w:], math.log(1e-30))


def test_target_orders_by_mean_mass():
    """For one head the target is monotone in F / N_t (log is increasing)."""
    S, w = 20, 2
    rng = np.random.default_rng(3)
    Fh = rng.random((1, S))
    r = oracle.kvpop_target(Fh, w, 1, eps=1e-12)[0]
    m = Fh[0] / np.maximum(1, S - (np.arange(S) + w))
    assert (np.argsort(r, kind="stable") == np.argsort(m, kind="stable")).all()
