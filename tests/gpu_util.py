"""Shared helpers of the GPU parity tests: tolerances and comparisons.

Tolerances:
* F (future-attention mass): max relative error 2e-3 over entries whose
  oracle value is > 0; entries the oracle gives exactly 0 (keys past S-1-w)
  must be exactly 0.
* LSE: absolute error 1e-3 (a natural-log offset error e shifts every
  probability of the row by the factor exp(e), i.e. a relative error ~e in F,
  so 1e-3 keeps F inside its 2e-3 budget).
* selection indices, counts and compacted K/V: bit-exact.
* decode output: max absolute error 2e-3; key mass: relative 2e-3 plus 1e-9.
* Soft-TopK ratios: relative 1e-12; budgets exact unless r*t lies within
  1e-9 of an integer (then either floor is accepted).
"""
import numpy as np
import torch

F_RTOL = 2e-3
LSE_ATOL = 1e-3
DECODE_ATOL = 2e-3


def np64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def check_F(F_gpu, F_ref, what=""):
    F_gpu = np.asarray(F_gpu, dtype=np.float64)
    F_ref = np.asarray(F_ref, dtype=np.float64)
    assert F_gpu.shape == F_ref.shape, (F_gpu.shape, F_ref.shape)
    pos = F_ref > 0
    zero = ~pos
    assert (F_gpu[zero] == 0).all(), f"{what}: nonzero F where the oracle is exactly 0"
    if pos.any():
        rel = np.abs(F_gpu[pos] - F_ref[pos]) / F_ref[pos]
        assert rel.max() <= F_RTOL, f"{what}: F max rel err {rel.max():.3e}"
        return float(rel.max())
    return 0.0


def check_lse(lse_gpu, lse_ref, what=""):
    err = np.abs(np.asarray(lse_gpu, np.float64) - np.asarray(lse_ref, np.float64)).max()
    assert err <= LSE_ATOL, f"{what}: lse max abs err {err:.3e}"
    return float(err)


def oracle_row_lse_threads(q, k, scale, rows_per_task=2048):
    """oracle.row_lse over all rows, the rows split across host threads (numpy releases the
    GIL in its matrix products and elementwise loops).  The oracle itself is unchanged: every
    task is one call of it on a range of rows; q, k are converted to fp64 numpy once."""
    import concurrent.futures as cf
    import os

    import oracle
    q = np64(q) if isinstance(q, torch.Tensor) else np.asarray(q, np.float64)
    k = np64(k) if isinstance(k, torch.Tensor) else np.asarray(k, np.float64)
    Hq, S, _ = q.shape
    G = Hq // k.shape[0]
    out = np.empty((Hq, S))
    tasks = [(h, r0) for h in range(Hq) for r0 in range(0, S, rows_per_task)]
    tasks.sort(key=lambda t: -t[1])           # longest rows first

    def run(t):
        h, r0 = t
        rows = np.arange(r0, min(S, r0 + rows_per_task))
        out[h, rows] = oracle.row_lse(q[h:h + 1], k[h // G:h // G + 1], scale, rows=rows)[0]

    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        list(ex.map(run, tasks))
    return out


def oracle_future_mass_threads(q, k, lse, scale, window, keys, keys_per_task=256):
    """oracle.future_attn_mass on the listed keys, split across host threads (one oracle call
    per key range)."""
    import concurrent.futures as cf
    import os

    import oracle
    q = np64(q) if isinstance(q, torch.Tensor) else np.asarray(q, np.float64)
    k = np64(k) if isinstance(k, torch.Tensor) else np.asarray(k, np.float64)
    keys = np.asarray(keys, np.int64)
    F = np.empty((k.shape[0], keys.size))
    spans = [(a, min(keys.size, a + keys_per_task)) for a in range(0, keys.size, keys_per_task)]

    def run(sp):
        a, b = sp
        F[:, a:b] = oracle.future_attn_mass(q, k, lse, scale, window, keys=keys[a:b])

    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        list(ex.map(run, spans))
    return F
