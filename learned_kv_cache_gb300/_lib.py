"""ctypes binding of libkvp.so: the C ABI of include/kvp.h under the same names.

Argument marshalling only: every function checks tensor devices, dtypes,
shapes and contiguity (Q/K of the attention passes may be strided views whose
head_dim axis is contiguous), passes raw device pointers, strides and the current CUDA stream
to the library, and raises :class:`KvpError` on a non-zero status.  All
arithmetic runs in the library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvp.so")

KVP_F32, KVP_BF16, KVP_F16 = 0, 1, 2
_DTYPE = {torch.float32: KVP_F32, torch.bfloat16: KVP_BF16, torch.float16: KVP_F16}

STATUS = {0: "KVP_OK", -1: "KVP_ERR_INVALID_ARG", -2: "KVP_ERR_UNSUPPORTED", -3: "KVP_ERR_CUDA",
          -4: "KVP_ERR_TIMEOUT", -5: "KVP_ERR_WORKSPACE", -6: "KVP_ERR_DEVICE_CHECK"}

# Exported symbols and their C signatures (restype, argtypes), mirroring include/kvp.h.
_P, _I, _F, _D, _SZ, _I64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double,
                             ctypes.c_size_t, ctypes.c_int64)
SIGNATURES = {
    "kvp_lse_pass": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _F, _P, _P]),
    "kvp_future_attn_mass_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "kvp_future_attn_mass": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _F, _I, _P, _P, _SZ, _P]),
    "kvp_future_attn_target_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "kvp_future_attn_target": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _F, _I, _F, _I, _P, _P, _P,
                                    _P, _SZ, _P]),
    "kvp_topk_cutoffs": (_I, [_P, _I, _I, _I, _I, _I, _P, _P]),
    "kvp_sparse_lse_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "kvp_sparse_lse_pass": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _F, _I, _I, _P, _P, _SZ,
                                 _P]),
    "kvp_soft_topk_budgets": (_I, [_P, _I, _D, _I, _P, _P, _P]),
    "kvp_select_topk": (_I, [_P, _I, _I, _I64, _P, _I, _I, _P, _I, _P, _P]),
    "kvp_compact_kv": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P]),
    "kvp_chunk_compress": (_I, [_P, _P, _P, _P, _I, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P,
                                _P, _P, _P, _P, _I, _P]),
    "kvp_rank_rows_workspace_size": (_SZ, [_I, _I]),
    "kvp_rank_rows": (_I, [_P, _I, _I, _P, _P, _SZ, _P]),
    "kvp_eviction_auc_workspace_size": (_SZ, [_I, _I, _I]),
    "kvp_eviction_auc": (_I, [_P, _P, _I, _I, _I, _P, _P, _SZ, _P]),
    "kvp_ring_insert": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _I, _I, _P, _P]),
    "kvp_decode_attn_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "kvp_decode_attn": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _F, _P, _P, _P, _I, _I, _P,
                             _SZ, _P]),
    "kvp_decode_attn_noalloc": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _F, _P, _P]),
    "kvp_status_string": (ctypes.c_char_p, [_I]),
    "kvp_last_error": (ctypes.c_char_p, []),
    "kvp_check_device_status": (_I, [_P]),
    "kvp_abi_version": (_I, []),
    "kvp_launch_count": (ctypes.c_uint64, []),
}


class KvpError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {STATUS.get(status, status)}: {msg}")
        self.status = status


_lib = None


def load(path: str = LIB_PATH):
    """Load libkvp.so (raises if it has not been built: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(fn, rc):
    if rc != 0:
        msg = load().kvp_last_error().decode(errors="replace")
        raise KvpError(fn, rc, msg)


def _need(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _dtype(t):
    if t.dtype not in _DTYPE:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return _DTYPE[t.dtype]


def _bhsd(q, k):
    """Accept [B,H,S,D] or [H,S,D] (B = 1)."""
    if q.dim() == 3:
        q, k = q.unsqueeze(0), k.unsqueeze(0)
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q/k must be [B,H,S,D] or [H,S,D]")
    return q, k


def _strided_input(t: torch.Tensor, name: str, dtype=None, shape=None):
    """A [B,H,S,D] Q/K view read in place: the head_dim axis must be contiguous; returns the
    {batch, head, token} element strides as a C int64[3] (None when the view is dense)."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.stride(3) != 1 and t.shape[3] > 1:
        raise ValueError(f"{name}: the head_dim axis must be contiguous")
    if t.is_contiguous():
        return None
    return (ctypes.c_int64 * 3)(t.stride(0), t.stride(1), t.stride(2))


def kvp_lse_pass(q, k, sm_scale=None, lse=None, stream=None):
    """Causal row LSE: q [B,H_q,S,D], k [B,H_kv,S,D] -> lse fp32 [B,H_q,S]."""
    squeeze = q.dim() == 3
    q4, k4 = _bhsd(q, k)
    B, Hq, S, D = q4.shape
    Hkv = k4.shape[1]
    qs = _strided_input(q4, "q")
    ks = _strided_input(k4, "k", dtype=q4.dtype, shape=(B, Hkv, S, D))
    if sm_scale is None:
        sm_scale = D ** -0.5
    if lse is None:
        lse = torch.empty(B, Hq, S, device=q.device, dtype=torch.float32)
    _need(lse, "lse", torch.float32)
    if lse.numel() != B * Hq * S:
        raise ValueError("lse has the wrong size")
    rc = load().kvp_lse_pass(_ptr(q4), _ptr(k4), _dtype(q4), B, Hq, Hkv, S, D, qs, ks, float(sm_scale),
                             _ptr(lse), _stream(stream))
    _check("kvp_lse_pass", rc)
    return lse[0] if squeeze and lse.dim() == 3 else lse


def kvp_topk_cutoffs(ranks, n_sink, window, k, tau=None, stream=None):
    """Running top-k cutoffs: ranks int32 [..., S] (one row per KV head) -> tau int32 [..., S]."""
    _need(ranks, "ranks", torch.int32)
    S = ranks.shape[-1]
    H = ranks.numel() // max(S, 1)
    if tau is None:
        tau = torch.empty_like(ranks)
    _need(tau, "tau", torch.int32, tuple(ranks.shape))
    rc = load().kvp_topk_cutoffs(_ptr(ranks), H, S, int(n_sink), int(window), int(k), _ptr(tau),
                                 _stream(stream))
    _check("kvp_topk_cutoffs", rc)
    return tau


def kvp_sparse_lse_workspace_size(dtype, n_batch, h_q, h_kv, seq_len, head_dim):
    dt = _DTYPE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(load().kvp_sparse_lse_workspace_size(dt, n_batch, h_q, h_kv, seq_len, head_dim))


def kvp_sparse_lse_pass(q, k, ranks, tau, n_sink, window, sm_scale=None, lse=None, workspace=None,
                        stream=None):
    """Sparse row LSE under the running top-k mask: q [B,H_q,S,D], k [B,H_kv,S,D], ranks and
    tau int32 [B,H_kv,S] -> lse fp32 [B,H_q,S]."""
    squeeze = q.dim() == 3
    q4, k4 = _bhsd(q, k)
    B, Hq, S, D = q4.shape
    Hkv = k4.shape[1]
    qs = _strided_input(q4, "q")
    ks = _strided_input(k4, "k", dtype=q4.dtype, shape=(B, Hkv, S, D))
    _need(ranks, "ranks", torch.int32)
    _need(tau, "tau", torch.int32)
    if ranks.numel() != B * Hkv * S or tau.numel() != B * Hkv * S:
        raise ValueError("ranks / tau must hold n_batch * h_kv * seq_len entries")
    if sm_scale is None:
        sm_scale = D ** -0.5
    if lse is None:
        lse = torch.empty(B, Hq, S, device=q.device, dtype=torch.float32)
    _need(lse, "lse", torch.float32)
    if lse.numel() != B * Hq * S:
        raise ValueError("lse has the wrong size")
    need = kvp_sparse_lse_workspace_size(_dtype(q4), B, Hq, Hkv, S, D)
    if workspace is None and need > 0:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().kvp_sparse_lse_pass(_ptr(q4), _ptr(k4), _ptr(ranks), _ptr(tau), _dtype(q4), B, Hq, Hkv,
                                    S, D, qs, ks, float(sm_scale), int(n_sink), int(window), _ptr(lse),
                                    _ptr(workspace), ws_bytes, _stream(stream))
    _check("kvp_sparse_lse_pass", rc)
    return lse[0] if squeeze and lse.dim() == 3 else lse


def kvp_future_attn_mass_workspace_size(dtype, n_batch, h_q, h_kv, seq_len, head_dim, window):
    dt = _DTYPE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(load().kvp_future_attn_mass_workspace_size(dt, n_batch, h_q, h_kv, seq_len,
                                                          head_dim, window))


def kvp_future_attn_mass(q, k, lse, window, sm_scale=None, F=None, workspace=None, stream=None):
    """Future-attention mass: -> F fp32 [B,H_kv,S] (raw group sum over queries i >= j + window)."""
    squeeze = q.dim() == 3
    q4, k4 = _bhsd(q, k)
    B, Hq, S, D = q4.shape
    Hkv = k4.shape[1]
    qs = _strided_input(q4, "q")
    ks = _strided_input(k4, "k", dtype=q4.dtype, shape=(B, Hkv, S, D))
    _need(lse, "lse", torch.float32)
    if lse.numel() != B * Hq * S:
        raise ValueError("lse has the wrong size")
    if sm_scale is None:
        sm_scale = D ** -0.5
    if F is None:
        F = torch.empty(B, Hkv, S, device=q.device, dtype=torch.float32)
    _need(F, "F", torch.float32)
    if F.numel() != B * Hkv * S:
        raise ValueError("F has the wrong size")
    need = kvp_future_attn_mass_workspace_size(q4.dtype, B, Hq, Hkv, S, D, int(window))
    if workspace is None and need > 0:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().kvp_future_attn_mass(_ptr(q4), _ptr(k4), _ptr(lse), _dtype(q4), B, Hq, Hkv, S, D,
                                     qs, ks, float(sm_scale), int(window), _ptr(F), _ptr(workspace),
                                     ws_bytes, _stream(stream))
    _check("kvp_future_attn_mass", rc)
    return F[0] if squeeze and F.dim() == 3 else F


KVP_TARGET_MAX_LOG, KVP_TARGET_MEAN_PROB = 0, 1


def kvp_future_attn_target_workspace_size(dtype, n_batch, h_q, h_kv, seq_len, head_dim, window):
    dt = _DTYPE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(load().kvp_future_attn_target_workspace_size(dt, n_batch, h_q, h_kv, seq_len,
                                                            head_dim, window))


def kvp_future_attn_target(q, k, lse, window, eps=0.0, aggregate="max_log", sm_scale=None,
                           target=None, F_heads=None, F=None, want=("target",), workspace=None,
                           stream=None):
    """KVpop target: returns (target [B,H_kv,S], F_heads [B,H_q,S] or None, F [B,H_kv,S] or None)."""
    q4, k4 = _bhsd(q, k)
    B, Hq, S, D = q4.shape
    Hkv = k4.shape[1]
    qs = _strided_input(q4, "q")
    ks = _strided_input(k4, "k", dtype=q4.dtype, shape=(B, Hkv, S, D))
    _need(lse, "lse", torch.float32)
    if sm_scale is None:
        sm_scale = D ** -0.5
    agg = {"max_log": KVP_TARGET_MAX_LOG, "mean_prob": KVP_TARGET_MEAN_PROB}[aggregate]
    dev = q.device
    if target is None and "target" in want:
        target = torch.empty(B, Hkv, S, device=dev, dtype=torch.float32)
    if F_heads is None and "F_heads" in want:
        F_heads = torch.empty(B, Hq, S, device=dev, dtype=torch.float32)
    if F is None and "F" in want:
        F = torch.empty(B, Hkv, S, device=dev, dtype=torch.float32)
    need = kvp_future_attn_target_workspace_size(_dtype(q4), B, Hq, Hkv, S, D, int(window))
    if workspace is None:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = load().kvp_future_attn_target(_ptr(q4), _ptr(k4), _ptr(lse), _dtype(q4), B, Hq, Hkv, S, D,
                                       qs, ks, float(sm_scale), int(window), float(eps), agg, _ptr(target),
                                       _ptr(F_heads), _ptr(F), _ptr(workspace), ws_bytes,
                                       _stream(stream))
    _check("kvp_future_attn_target", rc)
    return target, F_heads, F


def kvp_soft_topk_budgets(scores, k, t, ratios=None, budgets=None, stream=None):
    """Closed-form Soft-TopK ratios (fp64 [n]) and budgets floor(r*t) (int32 [n])."""
    _need(scores, "scores", torch.float64)
    n = scores.numel()
    if ratios is None:
        ratios = torch.empty(n, device=scores.device, dtype=torch.float64)
    if budgets is None:
        budgets = torch.empty(n, device=scores.device, dtype=torch.int32)
    _need(ratios, "ratios", torch.float64, (n,))
    _need(budgets, "budgets", torch.int32, (n,))
    rc = load().kvp_soft_topk_budgets(_ptr(scores), n, float(k), int(t), _ptr(ratios), _ptr(budgets),
                                      _stream(stream))
    _check("kvp_soft_topk_budgets", rc)
    return ratios, budgets


def kvp_select_topk(scores, budgets, n_sink, n_recent, b_max, T=None, idx=None, count=None,
                    stream=None):
    """scores fp32 [R, >=T] (row stride = scores.shape[1]) -> (idx int32 [R,b_max], count int32 [R])."""
    if scores.dim() != 2:
        raise ValueError("scores must be [R, T]")
    if not scores.is_cuda or scores.stride(1) != 1 or scores.dtype != torch.float32:
        raise ValueError("scores must be a CUDA fp32 tensor with unit column stride")
    R = scores.shape[0]
    T = scores.shape[1] if T is None else int(T)
    _need(budgets, "budgets", torch.int32, (R,))
    if idx is None:
        idx = torch.empty(R, b_max, device=scores.device, dtype=torch.int32)
    if count is None:
        count = torch.empty(R, device=scores.device, dtype=torch.int32)
    _need(idx, "idx", torch.int32, (R, b_max))
    _need(count, "count", torch.int32, (R,))
    rc = load().kvp_select_topk(_ptr(scores), R, T, scores.stride(0), _ptr(budgets), int(n_sink),
                                int(n_recent), _ptr(idx), int(b_max), _ptr(count), _stream(stream))
    _check("kvp_select_topk", rc)
    return idx, count


def kvp_compact_kv(k, v, idx, count, k_out=None, v_out=None, stream=None):
    """k, v [R,T,D] -> k_out, v_out [R,b_max,D] (rows m >= count[r] untouched)."""
    _need(k, "k")
    R, T, D = k.shape
    _need(v, "v", k.dtype, (R, T, D))
    b_max = idx.shape[1]
    _need(idx, "idx", torch.int32, (R, b_max))
    _need(count, "count", torch.int32, (R,))
    if k_out is None:
        k_out = torch.zeros(R, b_max, D, device=k.device, dtype=k.dtype)
    if v_out is None:
        v_out = torch.zeros(R, b_max, D, device=k.device, dtype=k.dtype)
    _need(k_out, "k_out", k.dtype, (R, b_max, D))
    _need(v_out, "v_out", k.dtype, (R, b_max, D))
    rc = load().kvp_compact_kv(_ptr(k), _ptr(v), _dtype(k), R, T, D, _ptr(idx), _ptr(count), b_max,
                               _ptr(k_out), _ptr(v_out), _stream(stream))
    _check("kvp_compact_kv", rc)
    return k_out, v_out


def kvp_chunk_compress(cache, n_in, chunk_k, chunk_v, chunk_score, pos0, budget, n_sink, n_recent,
                       out, idx=None, count=None, stream=None):
    """One chunked prefill-compress step.  ``cache`` and ``out`` are dicts of tensors "k", "v"
    [R, cap, D], "score" float32 [R, cap] and "pos" int32 [R, cap] (``cache`` may be None when
    n_in = 0).  Returns (idx, count)."""
    _need(chunk_k, "chunk_k")
    R, C, D = chunk_k.shape
    _need(chunk_v, "chunk_v", chunk_k.dtype, (R, C, D))
    _need(chunk_score, "chunk_score", torch.float32, (R, C))
    out_cap = out["k"].shape[1]
    _need(out["k"], "out k", chunk_k.dtype, (R, out_cap, D))
    _need(out["v"], "out v", chunk_k.dtype, (R, out_cap, D))
    _need(out["score"], "out score", torch.float32, (R, out_cap))
    _need(out["pos"], "out pos", torch.int32, (R, out_cap))
    if cache is not None:
        cap_in = cache["k"].shape[1]
        _need(cache["k"], "cache k", chunk_k.dtype, (R, cap_in, D))
        _need(cache["v"], "cache v", chunk_k.dtype, (R, cap_in, D))
        _need(cache["score"], "cache score", torch.float32, (R, cap_in))
        _need(cache["pos"], "cache pos", torch.int32, (R, cap_in))
        ck, cv, cs, cp = (_ptr(cache[x]) for x in ("k", "v", "score", "pos"))
    else:
        if n_in:
            raise ValueError("n_in > 0 needs a cache")
        cap_in, ck, cv, cs, cp = 0, None, None, None, None
    if idx is None:
        idx = torch.empty(R, out_cap, device=chunk_k.device, dtype=torch.int32)
    if count is None:
        count = torch.empty(R, device=chunk_k.device, dtype=torch.int32)
    _need(idx, "idx", torch.int32, (R, out_cap))
    _need(count, "count", torch.int32, (R,))
    rc = load().kvp_chunk_compress(ck, cv, cs, cp, cap_in, int(n_in), _ptr(chunk_k), _ptr(chunk_v),
                                   _ptr(chunk_score), C, int(pos0), _dtype(chunk_k), R, D, int(budget),
                                   int(n_sink), int(n_recent), _ptr(idx), _ptr(count), _ptr(out["k"]),
                                   _ptr(out["v"]), _ptr(out["score"]), _ptr(out["pos"]), out_cap,
                                   _stream(stream))
    _check("kvp_chunk_compress", rc)
    return idx, count


def kvp_rank_rows(scores, ranks=None, workspace=None, stream=None):
    """scores float32 [..., T] (one row per leading index) -> ranks int32 of the same shape."""
    _need(scores, "scores", torch.float32)
    T = scores.shape[-1]
    R = scores.numel() // max(T, 1)
    if ranks is None:
        ranks = torch.empty(scores.shape, device=scores.device, dtype=torch.int32)
    _need(ranks, "ranks", torch.int32, tuple(scores.shape))
    need = int(load().kvp_rank_rows_workspace_size(R, T))
    if workspace is None:
        workspace = torch.empty(need, device=scores.device, dtype=torch.uint8)
    rc = load().kvp_rank_rows(_ptr(scores), R, T, _ptr(ranks), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream))
    _check("kvp_rank_rows", rc)
    return ranks


def kvp_eviction_auc(F, ranks, auc=None, workspace=None, stream=None):
    """F float32 [R, T], ranks int32 [R, M, T] (or [R, T] for M = 1) -> auc float64 [R, M]."""
    _need(F, "F", torch.float32)
    R, T = F.shape
    r3 = ranks if ranks.dim() == 3 else ranks.unsqueeze(1)
    _need(r3, "ranks", torch.int32)
    if r3.shape[0] != R or r3.shape[2] != T:
        raise ValueError("ranks must be [R, M, T]")
    M = r3.shape[1]
    if auc is None:
        auc = torch.empty(R, M, device=F.device, dtype=torch.float64)
    _need(auc, "auc", torch.float64, (R, M))
    need = int(load().kvp_eviction_auc_workspace_size(R, M, T))
    if workspace is None:
        workspace = torch.empty(need, device=F.device, dtype=torch.uint8)
    rc = load().kvp_eviction_auc(_ptr(F), _ptr(r3), R, M, T, _ptr(auc), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream))
    _check("kvp_eviction_auc", rc)
    return auc


def kvp_ring_insert(kc, vc, slot_pos, slot_score, fill, new_k, new_v, new_pos, n_sink, n_recent,
                    out_slot=None, stream=None):
    """Insert one new token per row into a static cache [R, cap, D] in place (see kvp.h)."""
    _need(kc, "kc")
    R, cap, D = kc.shape
    _need(vc, "vc", kc.dtype, (R, cap, D))
    _need(slot_pos, "slot_pos", torch.int32, (R, cap))
    _need(slot_score, "slot_score", torch.float32, (R, cap))
    _need(fill, "fill", torch.int32, (R,))
    _need(new_k, "new_k", kc.dtype, (R, D))
    _need(new_v, "new_v", kc.dtype, (R, D))
    if out_slot is not None:
        _need(out_slot, "out_slot", torch.int32, (R,))
    rc = load().kvp_ring_insert(_ptr(kc), _ptr(vc), _ptr(slot_pos), _ptr(slot_score), _ptr(fill),
                                _dtype(kc), R, cap, D, _ptr(new_k), _ptr(new_v), int(new_pos),
                                int(n_sink), int(n_recent), _ptr(out_slot), _stream(stream))
    _check("kvp_ring_insert", rc)
    return out_slot


def kvp_decode_attn_workspace_size(n_layers, h_q, h_kv, head_dim, T_cap, with_key_mass):
    return int(load().kvp_decode_attn_workspace_size(n_layers, h_q, h_kv, head_dim, T_cap,
                                                     int(bool(with_key_mass))))


def kvp_decode_attn(q, kc, vc, lens, sm_scale=None, out=None, key_mass=None, key_pos=None,
                    T_src=None, accumulate=False, workspace=None, stream=None):
    """q [L,H_q,D]; kc, vc [L*H_kv,T_cap,D]; lens int32 [L*H_kv] -> out fp32 [L,H_q,D]."""
    _need(q, "q")
    L, Hq, D = q.shape
    R, T_cap, _ = kc.shape
    if R % L:
        raise ValueError("kc rows must be n_layers * h_kv")
    Hkv = R // L
    _need(kc, "kc", q.dtype, (R, T_cap, D))
    _need(vc, "vc", q.dtype, (R, T_cap, D))
    _need(lens, "lens", torch.int32, (R,))
    if sm_scale is None:
        sm_scale = D ** -0.5
    if out is None:
        out = torch.empty(L, Hq, D, device=q.device, dtype=torch.float32)
    _need(out, "out", torch.float32, (L, Hq, D))
    if key_mass is not None:
        _need(key_mass, "key_mass", torch.float32)
        T_src = key_mass.shape[1] if T_src is None else int(T_src)
        if key_pos is not None:
            _need(key_pos, "key_pos", torch.int32, (R, T_cap))
    need = kvp_decode_attn_workspace_size(L, Hq, Hkv, D, T_cap, key_mass is not None)
    if workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = load().kvp_decode_attn(_ptr(q), _ptr(kc), _ptr(vc), _dtype(q), L, Hq, Hkv, D, T_cap,
                                _ptr(lens), float(sm_scale), _ptr(out), _ptr(key_mass),
                                _ptr(key_pos), int(T_src or 0), int(bool(accumulate)),
                                _ptr(workspace), ws_bytes, _stream(stream))
    _check("kvp_decode_attn", rc)
    return out


def kvp_decode_attn_noalloc(q, kc, vc, lens, sm_scale=None, out=None, stream=None):
    """kvp_decode_attn without a workspace (the library's fixed per-device scratch is used
    instead); for callers that cannot allocate device memory.  Calls on one device must not
    overlap on the GPU."""
    _need(q, "q")
    L, Hq, D = q.shape
    R, T_cap, _ = kc.shape
    if R % L:
        raise ValueError("kc rows must be n_layers * h_kv")
    _need(kc, "kc", q.dtype, (R, T_cap, D))
    _need(vc, "vc", q.dtype, (R, T_cap, D))
    _need(lens, "lens", torch.int32, (R,))
    if sm_scale is None:
        sm_scale = D ** -0.5
    if out is None:
        out = torch.empty(L, Hq, D, device=q.device, dtype=torch.float32)
    _need(out, "out", torch.float32, (L, Hq, D))
    rc = load().kvp_decode_attn_noalloc(_ptr(q), _ptr(kc), _ptr(vc), _dtype(q), L, Hq, R // L, D,
                                        T_cap, _ptr(lens), float(sm_scale), _ptr(out),
                                        _stream(stream))
    _check("kvp_decode_attn_noalloc", rc)
    return out


def kvp_check_device_status(stream=None):
    rc = load().kvp_check_device_status(_stream(stream))
    _check("kvp_check_device_status", rc)


def kvp_abi_version():
    return int(load().kvp_abi_version())


def kvp_launch_count():
    return int(load().kvp_launch_count())
