"""fp64 oracle for learned head-wise budgets (LKV: End-to-End Learning of
Head-wise Budgets and Token Selection for LLM KV Cache Eviction).

"The Differentiable Soft-TopK Operator" prints only the threshold

    lambda = log( (sqrt((k-m)^2 + S1*S2) - (k-m)) / S1 ),
    S1 = sum_{i<=m} exp(-x_i),  S2 = sum_{i>m} exp(x_i)

over scores sorted descending, with m the number of scores at or above the
threshold, and states that the outputs sum to k, preserve order and are
translation invariant, and that the operator reduces to a softmax for k = 1.
The per-element map is not printed.  Reading taken here: each output is the
Laplace CDF of (x_i - lambda),

    r_i = 1 - exp(-(x_i - lambda)) / 2   if x_i >= lambda
    r_i =     exp(  x_i - lambda ) / 2   otherwise,

because setting sum_i r_i = k for this map and solving the resulting
quadratic in exp(lambda) gives exactly the printed threshold, and with m = 0
it gives r = k * softmax(x).  Temperature tau = 1.

The threshold is evaluated in the algebraically identical form
S2 / (sqrt((k-m)^2 + S1*S2) + (k-m)) when k - m >= 0, which avoids the
cancellation of the printed form and also covers m = 0 (S1 = 0).

"LKV-H: Learning Global Budget Allocation": ratios r = ST_{R_agg}(s) over the
flattened per-(layer, head) scores, and the discrete budget of a head is
b = floor(r * t).
"""
from __future__ import annotations

import numpy as np


def _threshold(S1: float, S2: float, k: float, m: int) -> float:
    a = k - m
    if a >= 0.0:
        return float(np.log(S2 / (np.sqrt(a * a + S1 * S2) + a)))
    return float(np.log((np.sqrt(a * a + S1 * S2) - a) / S1))


def soft_topk(x, k: float):
    """Returns (r fp64 [n], lambda) with sum(r) = k; requires 0 < k < n."""
    x = np.asarray(x, dtype=np.float64)
    n = x.size
    if not (0.0 < k < n):
        raise ValueError("need 0 < k < n")
    xs = np.sort(x)[::-1]
    e_neg = np.exp(-xs)
    e_pos = np.exp(xs)
    best_viol, lam = np.inf, None
    for m in range(n + 1):
        S1 = float(e_neg[:m].sum())
        S2 = float(e_pos[m:].sum())
        lam_m = _threshold(S1, S2, k, m)
        upper = xs[m - 1] if m > 0 else np.inf
        lower = xs[m] if m < n else -np.inf
        # the split is consistent when exactly the top m scores lie at or above the threshold;
        # the scores equal to it are a boundary where the neighbouring splits give the same r
        viol = max(0.0, lam_m - upper) + max(0.0, lower - lam_m)
        if viol < best_viol:
            best_viol, lam = viol, lam_m
        if viol == 0.0:
            break
    d = x - lam
    r = np.where(d >= 0.0, 1.0 - 0.5 * np.exp(-d), 0.5 * np.exp(np.minimum(d, 0.0)))
    return r, lam


def head_budgets(scores, retention: float, t: int):
    """LKV-H: r = ST_{R_agg}(s) with R_agg = retention * n, b = floor(r * t)."""
    s = np.asarray(scores, dtype=np.float64)
    r, lam = soft_topk(s, retention * s.size)
    b = np.floor(r * t).astype(np.int64)
    return r, b, lam
