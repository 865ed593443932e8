"""fp64 oracle for single-token decode attention over a (pruned) cache.

How much KV cache can you prune before quality degrades, "What we did" and
"Bounded windows: memory and decode-time impact": each decode step runs
one-token attention over the retained entries only; KVpop, Figure 1: attention
is computed over the retained set.  With the query q of head h_q and the
``len`` retained keys/values of its KV head:

    out = sum_m softmax_m(scale * q . Kc[m]) * Vc[m]

An empty row (len = 0) yields a zero output.  The optional key mass is the
group-summed probability each retained key receives (the cumulative
past-attention score of the blog's attention-score policy), scattered to the
key's source position.
"""
from __future__ import annotations

import numpy as np

from .attention_mass import _as_f64


def decode_attn(q, kc, vc, lens, scale: float, key_pos=None, T_src: int | None = None):
    """q [L, H_q, D]; kc, vc [L*H_kv, Tcap, D]; lens [L*H_kv].

    Returns (out [L, H_q, D] fp64, key_mass [L*H_kv, T_src] fp64 or None).
    ``key_pos`` [L*H_kv, Tcap] maps retained slot m to its source position
    (identity when None).
    """
    q = _as_f64(q)
    kc = _as_f64(kc)
    vc = _as_f64(vc)
    L, Hq, D = q.shape
    R, Tcap, _ = kc.shape
    Hkv = R // L
    G = Hq // Hkv
    lens = np.asarray(lens, dtype=np.int64)
    out = np.zeros((L, Hq, D))
    T_src = Tcap if T_src is None else int(T_src)
    mass = np.zeros((R, T_src))
    for l in range(L):
        for hq in range(Hq):
            r = l * Hkv + hq // G
            n = int(lens[r])
            if n == 0:
                continue
            s = (kc[r, :n] @ q[l, hq]) * scale
            m = s.max()
            e = np.exp(s - m)
            p = e / e.sum()
            out[l, hq] = p @ vc[r, :n]
            pos = np.arange(n) if key_pos is None else np.asarray(key_pos[r, :n], dtype=np.int64)
            np.add.at(mass[r], pos, p)
    return out, mass
