"""Seeded synthetic inputs shared by the CUDA path, the oracle and the benchmark.

The recipe (fixed draw order: Q, K, V, key scales, planted positions, decode
query) stands in for the real model activations the pages measured on; it
holds none of the method's arithmetic.  All values are drawn in fp32 and then
rounded (round-to-nearest-even) to the workload's storage dtype, so the
oracle and the kernels read bit-identical tensors.

* Q, K, V ~ N(0, 1).
* Per-KV-head key scale c_h ~ U[lo, hi] multiplies that head's keys.
* Sink keys: the first ``n_sink_keys`` tokens of every KV head get the key
  3 * sqrt(D) * qbar / |qbar|, with qbar the mean query of the head's group
  (the "mean query direction x3" construction).
* Retrieval keys: ``n_retrieval`` positions p ~ U[n_sink_keys, S-1-w) per KV
  head get the key of a later query, k_p := q_{h*G, i} with i ~ U[p+w, S-1].
* One decode query per query head ~ N(0, 1).
"""
from __future__ import annotations

import math

import torch

from .configs import Workload

_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def torch_dtype(name: str) -> torch.dtype:
    return _DT[name]


def _generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_prefill_layer(w: Workload, layer: int = 0, device="cpu", seq_len: int | None = None):
    """One layer of a prefill workload: dict with q [H_q,S,D], k/v [H_kv,S,D], dq [H_q,D]."""
    S = w.seq_len if seq_len is None else int(seq_len)
    Hq, Hkv, D, G = w.h_q, w.h_kv, w.head_dim, w.group
    gen = _generator(w.seed * 1000 + layer, device)
    f32 = torch.float32
    q = torch.randn(Hq, S, D, generator=gen, device=device, dtype=f32)
    k = torch.randn(Hkv, S, D, generator=gen, device=device, dtype=f32)
    v = torch.randn(Hkv, S, D, generator=gen, device=device, dtype=f32)
    if w.key_scale is not None:
        lo, hi = w.key_scale
        c = torch.rand(Hkv, generator=gen, device=device, dtype=f32) * (hi - lo) + lo
        k.mul_(c[:, None, None])
    if w.n_sink_keys > 0:
        ns = min(w.n_sink_keys, S)
        for h in range(Hkv):
            qbar = q[h * G:(h + 1) * G].reshape(-1, D).mean(dim=0)
            sink = qbar * (3.0 * math.sqrt(D) / qbar.norm())
            k[h, :ns] = sink
    if w.n_retrieval > 0:
        lo = w.n_sink_keys
        hi = S - 1 - w.window
        if hi > lo:
            for h in range(Hkv):
                pos = torch.randint(lo, hi, (w.n_retrieval,), generator=gen, device=device)
                u = torch.rand(w.n_retrieval, generator=gen, device=device, dtype=torch.float64)
                for t in range(w.n_retrieval):
                    p = int(pos[t])
                    first, last = p + w.window, S - 1
                    i = first + min(int(float(u[t]) * (last - first + 1)), last - first)
                    k[h, p] = q[h * G, i]
    dq = torch.randn(Hq, D, generator=gen, device=device, dtype=f32)
    dt = _DT[w.dtype]
    return {"q": q.to(dt), "k": k.to(dt), "v": v.to(dt), "dq": dq.to(dt)}


def make_prefill(w: Workload, device="cpu", seq_len: int | None = None, layers=None):
    """All (or the listed) layers stacked: q [L,H_q,S,D], k/v [L,H_kv,S,D], dq [L,H_q,D]."""
    layers = range(w.n_layers) if layers is None else list(layers)
    parts = [make_prefill_layer(w, l, device=device, seq_len=seq_len) for l in layers]
    return {key: torch.stack([p[key] for p in parts]) for key in parts[0]}


def make_decode_cache(w: Workload, device="cpu", seq_len: int | None = None):
    """Decode-eviction workload: k/v caches [L*H_kv, T, D], decode query q [L, H_q, D]."""
    T = w.seq_len if seq_len is None else int(seq_len)
    R, D = w.n_layers * w.h_kv, w.head_dim
    gen = _generator(w.seed * 1000, device)
    dt = _DT[w.dtype]
    f32 = torch.float32
    k = torch.randn(R, T, D, generator=gen, device=device, dtype=f32).to(dt)
    v = torch.randn(R, T, D, generator=gen, device=device, dtype=f32).to(dt)
    q = torch.randn(w.n_layers, w.h_q, D, generator=gen, device=device, dtype=f32).to(dt)
    return {"k": k, "v": v, "q": q}


def make_head_scores(n: int, seed: int, device="cpu") -> torch.Tensor:
    """Seeded N(0,1) head-importance scores (fp64) standing in for learned head scores."""
    gen = _generator(seed, device)
    return torch.randn(n, generator=gen, device=device, dtype=torch.float64)


def make_scores(R: int, T: int, seed: int, device="cpu", quantize: int | None = None,
                specials: bool = False) -> torch.Tensor:
    """Seeded fp32 score rows for selection tests.  ``quantize`` rounds to that many levels
    (heavy ties); ``specials`` plants -0.0, +0.0, +-inf and NaN values."""
    gen = _generator(seed, device)
    s = torch.randn(R, T, generator=gen, device=device, dtype=torch.float32)
    if quantize:
        s = torch.round(s * quantize) / quantize
    if specials and T >= 16:
        idx = torch.randint(0, T, (R, 12), generator=gen, device=device)
        vals = torch.tensor([-0.0, 0.0, float("inf"), float("-inf"), float("nan"), -0.0,
                             0.0, float("nan"), 1.0, 1.0, -1.0, float("inf")],
                            device=device, dtype=torch.float32)
        s.scatter_(1, idx, vals.expand(R, 12).contiguous())
    return s


def make_static_ranks(H: int, S: int, seed: int, device="cpu") -> torch.Tensor:
    """Seeded static token ranks: one random permutation of 0..S-1 per KV head (int32 [H, S]),
    standing in for the ranks a trained scorer's static priorities would give."""
    gen = _generator(seed, device)
    return torch.stack([torch.randperm(S, generator=gen, device=device) for _ in range(H)]).to(torch.int32)
