"""Pins of the chunked prefill-compress oracle.

With per-token scores that never change, a token evicted at some step was outside the top-k of
the tokens competing then, and every token that beat it is still kept later, so it would lose
the final competition as well: compressing chunk by chunk keeps exactly the tokens that one
selection over the whole prefix keeps (the sinks, the last n_recent tokens and the top-scoring
rest), whatever the chunk length.  The tests check that, plus the per-step invariants (count,
ascending source positions, sinks and the most recent tokens always kept, scores carried with
their tokens), including chunks shorter than the recent window and heavy score ties."""
import numpy as np
import pytest

from oracle.chunked import chunk_compress_step, chunked_prefill_compress
from oracle.selection import effective_budget, select_row


def _inputs(R, S, D, seed, ties=False):
    rng = np.random.default_rng(seed)
    k = rng.integers(-30000, 30000, (R, S, D)).astype(np.int16)
    v = rng.integers(-30000, 30000, (R, S, D)).astype(np.int16)
    s = rng.standard_normal((R, S)).astype(np.float32)
    if ties:
        s = np.round(s * 2).astype(np.float32) / 2
    return k, v, s


@pytest.mark.parametrize("S,C,b,ns,nr,ties", [
    (300, 64, 50, 4, 16, False), (300, 7, 50, 4, 16, False), (257, 300, 40, 2, 8, False),
    (500, 33, 120, 0, 1, True), (200, 50, 10, 4, 16, False), (400, 100, 64, 4, 64, True),
])
def test_chunked_equals_one_selection_over_the_prefix(S, C, b, ns, nr, ties):
    R, D = 3, 4
    k, v, s = _inputs(R, S, D, seed=S + C, ties=ties)
    cache, counts = chunked_prefill_compress(k, v, s, C, b, ns, nr)
    for r in range(R):
        keep = select_row(s[r].astype(np.float64), b, ns, nr)
        n = keep.size
        assert counts[-1] == n
        assert (cache["pos"][r, :n] == keep).all()
        assert (cache["k"][r, :n] == k[r, keep]).all() and (cache["v"][r, :n] == v[r, keep]).all()
        assert (cache["score"][r, :n] == s[r, keep]).all()


def test_step_invariants():
    R, S, D, C, b, ns, nr = 2, 260, 4, 40, 48, 4, 20
    k, v, s = _inputs(R, S, D, seed=9)
    cache, n = None, 0
    for p0 in range(0, S, C):
        p1 = min(S, p0 + C)
        cache, idx, cnt = chunk_compress_step(cache, n, k[:, p0:p1], v[:, p0:p1], s[:, p0:p1], p0, b, ns, nr)
        T = n + (p1 - p0)
        assert (cnt == effective_budget(T, b, ns, nr)).all()
        n = int(cnt[0])
        for r in range(R):
            pos = cache["pos"][r, :n]
            assert (np.diff(pos) > 0).all()
            assert set(range(min(ns, p1))) <= set(pos.tolist())
            assert set(range(max(0, p1 - nr), p1)) <= set(pos.tolist())
            assert (cache["score"][r, :n] == s[r, pos]).all()
            assert (idx[r, :n] < T).all() and (idx[r, n:] == -1).all()
