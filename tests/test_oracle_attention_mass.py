"""Pins of the fp64 oracle's row LSE and future-attention mass (no GPU).

Each check ties the oracle to something other than itself: brute force
through scipy softmax/logsumexp on tiny inputs, the uniform-attention closed
form, a hand-derived two-token case, and the invariants the definition fixes.
"""
import math

import numpy as np
import pytest

import oracle
from tests import brute


def _rand(Hq, Hkv, S, D, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((Hq, S, D)), rng.standard_normal((Hkv, S, D))


@pytest.mark.parametrize("Hq,Hkv,S,D,w", [(1, 1, 17, 8, 0), (2, 1, 33, 16, 3), (6, 2, 40, 8, 7),
                                          (4, 4, 25, 4, 1), (3, 1, 31, 8, 30), (2, 1, 29, 8, 29)])
def test_matches_brute_force(Hq, Hkv, S, D, w):
    q, k = _rand(Hq, Hkv, S, D, seed=S * 7 + w)
    scale = 1.0 / math.sqrt(D)
    lse = oracle.row_lse(q, k, scale)
    np.testing.assert_allclose(lse, brute.lse(q, k, scale), rtol=0, atol=1e-12)
    F = oracle.future_attn_mass(q, k, lse, scale, w)
    np.testing.assert_allclose(F, brute.future_mass(q, k, scale, w), rtol=1e-12, atol=1e-13)


def _harmonic(n):
    return sum(1.0 / m for m in range(1, n + 1))


@pytest.mark.parametrize("zero", ["k", "q"])
@pytest.mark.parametrize("S,w,G", [(16, 0, 1), (23, 4, 3), (64, 16, 2)])
def test_uniform_attention_closed_form(zero, S, w, G):
    """q.k = 0 everywhere: p_ij = 1/(i+1), so lse_i = ln(i+1) and
    F[j] = G * (H_S - H_{j+w}) for j <= S-1-w, else 0."""
    rng = np.random.default_rng(S)
    D = 8
    q = rng.standard_normal((G, S, D))
    k = rng.standard_normal((1, S, D))
    if zero == "k":
        k[:] = 0
    else:
        q[:] = 0
    lse = oracle.row_lse(q, k, 0.3)
    np.testing.assert_allclose(lse, np.log(np.arange(1, S + 1))[None].repeat(G, 0), atol=1e-13)
    F = oracle.future_attn_mass(q, k, lse, 0.3, w)[0]
    want = [G * (_harmonic(S) - _harmonic(j + w)) if j <= S - 1 - w else 0.0 for j in range(S)]
    np.testing.assert_allclose(F, want, rtol=1e-12, atol=1e-14)


def test_two_token_hand_derivation():
    """S = 2, D = 1, scale 1: lse_0 = a0 b0, lse_1 = ln(e^{a1 b0} + e^{a1 b1});
    at w = 0: F[0] = 1 + e^{a1 b0} / (e^{a1 b0} + e^{a1 b1}), F[1] = e^{a1 b1} / (...).
    Swapping q and k (a transposed operand) changes every value."""
    a0, a1, b0, b1 = 0.7, -1.3, 2.1, 0.4
    q = np.array([[[a0], [a1]]])
    k = np.array([[[b0], [b1]]])
    lse = oracle.row_lse(q, k, 1.0)
    z = math.exp(a1 * b0) + math.exp(a1 * b1)
    np.testing.assert_allclose(lse[0], [a0 * b0, math.log(z)], atol=1e-15)
    F = oracle.future_attn_mass(q, k, lse, 1.0, 0)[0]
    np.testing.assert_allclose(F, [1 + math.exp(a1 * b0) / z, math.exp(a1 * b1) / z], atol=1e-15)
    F1 = oracle.future_attn_mass(q, k, lse, 1.0, 1)[0]
    np.testing.assert_allclose(F1, [math.exp(a1 * b0) / z, 0.0], atol=1e-15)


def test_invariants():
    """At w = 0 every query distributes mass 1 over its visible keys: sum_j F = G*S.
    F >= 0, F[j] <= G*(S-j-w), and keys after S-1-w receive nothing."""
    G, S, D = 3, 48, 16
    q, k = _rand(G, 1, S, D, seed=5)
    q *= 2.0
    lse = oracle.row_lse(q, k, 1 / 4)
    F0 = oracle.future_attn_mass(q, k, lse, 1 / 4, 0)[0]
    assert abs(F0.sum() - G * S) < 1e-10
    for w in (1, 5, S - 1):
        F = oracle.future_attn_mass(q, k, lse, 1 / 4, w)[0]
        assert (F >= 0).all()
        j = np.arange(S)
        assert (F <= G * np.maximum(S - j - w, 0) + 1e-12).all()
        assert (F[S - w:] == 0).all()


def test_last_window_only_key0():
    """w = S-1: only key 0 is past the window, for query S-1 alone: F[0] = sum_g p_{S-1,0}."""
    G, S, D = 2, 12, 4
    q, k = _rand(G, 1, S, D, seed=9)
    lse = oracle.row_lse(q, k, 0.5)
    F = oracle.future_attn_mass(q, k, lse, 0.5, S - 1)[0]
    want = sum(math.exp(0.5 * q[g, S - 1] @ k[0, 0] - lse[g, S - 1]) for g in range(G))
    assert abs(F[0] - want) < 1e-14
    assert (F[1:] == 0).all()


def test_single_token():
    """S = 1: lse = s_00 and at w = 0 the key gets mass G."""
    q = np.array([[[1.5, -2.0]], [[0.25, 1.0]]])
    k = np.array([[[0.5, 0.75]]])
    lse = oracle.row_lse(q, k, 0.7)
    np.testing.assert_allclose(lse[:, 0], 0.7 * (q[:, 0] @ k[0, 0]), atol=1e-15)
    F = oracle.future_attn_mass(q, k, lse, 0.7, 0)
    np.testing.assert_allclose(F, [[2.0]], atol=1e-15)


def test_row_and_key_subsets_agree_with_full():
    Hq, Hkv, S, D, w = 4, 2, 70, 8, 6
    q, k = _rand(Hq, Hkv, S, D, seed=11)
    lse = oracle.row_lse(q, k, 0.35)
    rows = np.array([69, 0, 33, 5])
    np.testing.assert_allclose(oracle.row_lse(q, k, 0.35, rows=rows), lse[:, rows], atol=1e-13)
    keys = np.array([63, 64, 0, 17, 69])
    F = oracle.future_attn_mass(q, k, lse, 0.35, w)
    np.testing.assert_allclose(oracle.future_attn_mass(q, k, lse, 0.35, w, keys=keys), F[:, keys],
                               rtol=1e-13, atol=1e-15)
