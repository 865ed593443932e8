"""Pins of the ring-cache oracle (no GPU): hand-worked steps, the blog's policy invariants
over a long simulation, and agreement with one-shot selection when scores are frozen."""
import numpy as np
import pytest

import oracle


def test_hand_worked_steps():
    # cap 6, 1 sink, 2 newest protected; slots hold tokens 0..5, new token 6
    pos = np.array([0, 1, 2, 3, 4, 5])
    score = np.array([9.0, 0.5, 0.2, 0.7, 0.2, 0.1])
    # evictable: 1 <= p <= 6 - 2 = 4 -> tokens 1..4; lowest score 0.2 at tokens 2 and 4 -> the newer (4)
    assert oracle.ring_victim(pos, score, 6, 6, 6, 1, 2) == 4
    # not full: append
    assert oracle.ring_victim(pos, score, 3, 6, 6, 1, 2) == 3
    # token 5 is the lowest but protected by the window; with a window of 1 it goes
    assert oracle.ring_victim(pos, score, 6, 6, 6, 1, 1) == 5
    # NaN is evicted first, -0.0 ties with +0.0
    assert oracle.ring_victim(pos, np.array([9, 0.5, np.nan, 0.7, 0.2, 0.1]), 6, 6, 6, 1, 2) == 2
    assert oracle.ring_victim(pos, np.array([9, -0.0, 0.0, 0.7, 0.2, 0.1]), 6, 6, 6, 1, 2) == 2
    # nothing evictable
    assert oracle.ring_victim(pos, score, 6, 6, 6, 3, 4) == -1


def test_insert_writes_slot_and_resets_score():
    R, cap, D = 2, 4, 3
    kc = np.zeros((R, cap, D)); vc = np.zeros((R, cap, D))
    pos = np.array([[0, 1, 2, 3], [0, 1, 2, -1]])
    score = np.array([[5.0, 1.0, 3.0, 4.0], [1.0, 2.0, 3.0, 0.0]])
    fill = np.array([4, 3])
    nk = np.arange(R * D, dtype=float).reshape(R, D)
    slots = oracle.ring_insert(kc, vc, pos, score, fill, nk, -nk, 4, 1, 1)
    assert slots.tolist() == [1, 3]
    assert (kc[0, 1] == nk[0]).all() and (vc[1, 3] == -nk[1]).all()
    assert pos[0, 1] == 4 and score[0, 1] == 0.0 and fill.tolist() == [4, 4]


def test_policy_invariants_over_a_stream():
    """Sinks and the newest n_recent tokens are always cached, the cache never exceeds its
    capacity, and every token ever evicted had the lowest score among the evictable ones."""
    rng = np.random.default_rng(0)
    cap, n_sink, n_recent, steps = 12, 2, 3, 200
    pos = np.full(cap, -1); score = np.zeros(cap); fill = 0
    for t in range(steps):
        live = pos[:fill]
        score[:fill] += rng.random(fill)                     # this step's attention
        m = oracle.ring_victim(pos, score, fill, cap, t, n_sink, n_recent)
        if fill == cap:
            ev = [s for s in range(cap) if n_sink <= pos[s] <= t - n_recent]
            assert score[m] == min(score[s] for s in ev)
        pos[m] = t; score[m] = 0.0; fill = min(cap, fill + 1)
        cached = set(pos[:fill].tolist())
        assert set(range(min(n_sink, t + 1))) <= cached
        assert set(range(max(0, t - n_recent + 1), t + 1)) <= cached
        assert fill <= cap


def test_frozen_scores_match_one_shot_selection():
    """With static per-token scores (no accumulation) streaming through the ring keeps the same
    set as the one-shot selection of the whole history when the low scorers are already old:
    here scores grow with position so every eviction removes the oldest evictable token."""
    cap, n_sink, n_recent, T = 8, 2, 2, 30
    tok_score = np.arange(T, dtype=float)
    pos = np.full(cap, -1); score = np.zeros(cap); fill = 0
    for t in range(T):
        for s in range(fill):
            score[s] = tok_score[pos[s]]
        m = oracle.ring_victim(pos, score, fill, cap, t, n_sink, n_recent)
        pos[m] = t; score[m] = tok_score[t]; fill = min(cap, fill + 1)
    want = oracle.select_row(tok_score, cap, n_sink, n_recent)
    assert sorted(pos.tolist()) == want.tolist()
