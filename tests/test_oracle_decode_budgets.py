"""Pins of the decode and Soft-TopK oracles (no GPU)."""
import math

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from tests import brute


def test_decode_matches_scipy_softmax():
    rng = np.random.default_rng(0)
    L, Hq, Hkv, T, D = 2, 6, 2, 37, 16
    q = rng.standard_normal((L, Hq, D))
    kc = rng.standard_normal((L * Hkv, T, D))
    vc = rng.standard_normal((L * Hkv, T, D))
    lens = np.array([37, 5, 1, 20])
    out, mass = oracle.decode_attn(q, kc, vc, lens, 0.25)
    G = Hq // Hkv
    for l in range(L):
        for h in range(Hq):
            r = l * Hkv + h // G
            want, _ = brute.decode(q[l, h], kc[r, :lens[r]], vc[r, :lens[r]], 0.25)
            np.testing.assert_allclose(out[l, h], want, atol=1e-13)
    # every query head distributes mass 1 over the kept keys of its KV head
    np.testing.assert_allclose(mass.sum(axis=1), G, atol=1e-12)


def test_decode_single_key_and_identical_keys():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 2, 8))
    kc = np.repeat(rng.standard_normal((1, 1, 8)), 9, axis=1)
    vc = rng.standard_normal((1, 9, 8))
    out, _ = oracle.decode_attn(q, kc, vc, [1], 0.5)
    np.testing.assert_allclose(out[0], vc[0, [0, 0]], atol=1e-15)
    out, _ = oracle.decode_attn(q, kc, vc, [9], 0.5)
    np.testing.assert_allclose(out[0], vc[0].mean(axis=0)[None].repeat(2, 0), atol=1e-14)


def test_decode_empty_row_is_zero():
    out, mass = oracle.decode_attn(np.ones((1, 1, 4)), np.ones((1, 3, 4)), np.ones((1, 3, 4)), [0], 1.0)
    assert not out.any() and not mass.any()


def test_compacted_decode_equals_masked_full_decode():
    """Learning to Evict, §A.2: eviction by an attention mask and by physical compaction
    are the same computation."""
    rng = np.random.default_rng(2)
    T, D = 64, 8
    k = rng.standard_normal((1, T, D))
    v = rng.standard_normal((1, T, D))
    q = rng.standard_normal((1, 1, D))
    idx, count = oracle.select_topk(rng.standard_normal((1, T)), [20], 4, 8)
    kc, vc = oracle.compact_kv(k, v, idx, count)
    out, mass = oracle.decode_attn(q, kc, vc, count, 0.3, key_pos=idx, T_src=T)
    logits = (k[0] @ q[0, 0]) * 0.3
    keep = np.zeros(T, bool)
    keep[idx[0, :20]] = True
    p = softmax(np.where(keep, logits, -np.inf))
    np.testing.assert_allclose(out[0, 0], p @ v[0], atol=1e-13)
    np.testing.assert_allclose(mass[0], p, atol=1e-14)


def _laplace_r(x, lam):
    d = x - lam
    return np.where(d >= 0, 1 - 0.5 * np.exp(-d), 0.5 * np.exp(np.minimum(d, 0)))


def _bisect_threshold(x, k):
    lo, hi = x.min() - 60.0, x.max() + 60.0
    for _ in range(300):
        mid = 0.5 * (lo + hi)
        if _laplace_r(x, mid).sum() > k:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


@pytest.mark.parametrize("n,k,seed", [(256, 38.4, 0), (10, 3.0, 1), (7, 6.5, 2), (50, 0.3, 3), (256, 200.0, 4)])
def test_soft_topk_threshold_solves_budget_equation(n, k, seed):
    """The printed closed-form threshold (LKV, "The Differentiable Soft-TopK Operator") must
    be the root of sum_i r_i(lambda) = k, found here independently by bisection."""
    x = np.random.default_rng(seed).standard_normal(n) * 1.5
    r, lam = oracle.soft_topk(x, k)
    assert abs(lam - _bisect_threshold(x, k)) < 1e-9
    assert abs(r.sum() - k) < 1e-11
    assert ((r > 0) & (r < 1)).all()


def test_soft_topk_order_and_translation():
    x = np.random.default_rng(5).standard_normal(100)
    r, lam = oracle.soft_topk(x, 20.0)
    o = np.argsort(x)
    assert (np.diff(r[o]) >= 0).all()
    r2, lam2 = oracle.soft_topk(x + 3.75, 20.0)
    np.testing.assert_allclose(r2, r, atol=1e-13)
    assert abs(lam2 - lam - 3.75) < 1e-12


def test_soft_topk_reduces_to_softmax():
    """When every score lies below the threshold (m = 0) the operator is k * softmax."""
    x = np.random.default_rng(6).standard_normal(64) * 0.1
    r, lam = oracle.soft_topk(x, 1.0)
    assert lam > x.max()
    np.testing.assert_allclose(r, softmax(x), rtol=1e-12)


def test_soft_topk_hard_limit():
    """Sharp scores (small temperature) approach the hard top-k indicator.  Distinct integer
    scores at temperature 0.05 keep every exponent inside the fp64 range."""
    x = np.random.default_rng(7).permutation(30).astype(np.float64)
    r, _ = oracle.soft_topk(x / 0.05, 5.0)
    want = np.zeros(30)
    want[np.argsort(-x)[:5]] = 1
    np.testing.assert_allclose(r, want, atol=0.5 * np.exp(-0.5 / 0.05) * 1.01)  # half-gap bound


def test_head_budgets_floor():
    s = np.random.default_rng(8).standard_normal(256)
    r, b, _ = oracle.head_budgets(s, 0.15, 32768)
    assert abs(r.sum() - 38.4) < 1e-10
    assert (b == np.floor(r * 32768)).all()
    assert b.min() > 4 + 64          # sinks + window always fit for this recipe
