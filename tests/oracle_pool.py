"""Host process pool that runs oracle calls in parallel for the full-size parity tests.

Test infrastructure.  It adds no arithmetic of its own: every task is one call of an oracle
function (``oracle.row_lse`` on a range of rows, ``oracle.future_attn_mass`` on a range of
keys) and the results are placed side by side.  Workers are spawned (never forked from a
process that has initialised CUDA), run one BLAS thread each and read the fp64 inputs through
memory maps of .npy files, so a few GB of inputs are written once and shared by every worker.
This module imports only numpy and the oracle.
"""
from __future__ import annotations

import contextlib
import multiprocessing as mp
import os
import tempfile

import numpy as np

_Q = None
_K = None


def _init(qpath, kpath):
    global _Q, _K
    _Q = np.load(qpath, mmap_mode="r")
    _K = np.load(kpath, mmap_mode="r")


def _lse_task(args):
    import oracle
    h, r0, r1, scale = args
    G = _Q.shape[0] // _K.shape[0]
    rows = np.arange(r0, r1)
    return h, r0, oracle.row_lse(_Q[h:h + 1], _K[h // G:h // G + 1], scale, rows=rows)[0]


def _mass_task(args):
    import oracle
    a, keys, lse, scale, window = args
    return a, oracle.future_attn_mass(_Q, _K, lse, scale, window, keys=keys)


@contextlib.contextmanager
def _single_thread_blas():
    names = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {n: os.environ.get(n) for n in names}
    for n in names:
        os.environ[n] = "1"
    try:
        yield
    finally:
        for n, v in saved.items():
            if v is None:
                os.environ.pop(n, None)
            else:
                os.environ[n] = v


class OraclePool:
    """``with OraclePool(q, k) as pool:`` -- q [H_q, S, D], k [H_kv, S, D] (fp64 numpy)."""

    def __init__(self, q, k, workers: int | None = None):
        self.q = np.ascontiguousarray(q, dtype=np.float64)
        self.k = np.ascontiguousarray(k, dtype=np.float64)
        self.workers = workers or os.cpu_count() or 4

    def __enter__(self):
        self._dir = tempfile.TemporaryDirectory(prefix="kvp_oracle_")
        qp = os.path.join(self._dir.name, "q.npy")
        kp = os.path.join(self._dir.name, "k.npy")
        np.save(qp, self.q)
        np.save(kp, self.k)
        with _single_thread_blas():
            self._pool = mp.get_context("spawn").Pool(self.workers, initializer=_init, initargs=(qp, kp))
        return self

    def __exit__(self, *exc):
        self._pool.close()
        self._pool.join()
        self._dir.cleanup()

    def row_lse(self, scale: float, rows_per_task: int = 1024) -> np.ndarray:
        """oracle.row_lse over every row of every query head."""
        Hq, S, _ = self.q.shape
        tasks = [(h, r0, min(S, r0 + rows_per_task), scale)
                 for r0 in range(0, S, rows_per_task) for h in range(Hq)]
        tasks.sort(key=lambda t: -t[1])                 # longest rows first
        out = np.empty((Hq, S))
        for h, r0, vals in self._pool.imap_unordered(_lse_task, tasks):
            out[h, r0:r0 + vals.size] = vals
        return out

    def future_attn_mass(self, lse, scale: float, window: int, keys, keys_per_task: int = 64):
        """oracle.future_attn_mass on the listed keys."""
        keys = np.asarray(keys, np.int64)
        lse = np.asarray(lse, np.float64)
        tasks = [(a, keys[a:a + keys_per_task], lse, scale, window)
                 for a in range(0, keys.size, keys_per_task)]
        F = np.empty((self.k.shape[0], keys.size))
        for a, vals in self._pool.imap_unordered(_mass_task, tasks):
            F[:, a:a + vals.shape[1]] = vals
        return F
