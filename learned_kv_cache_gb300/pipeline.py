"""One pass of the whole hot path with preallocated device buffers.

prefill K/V  ->  row LSE  ->  future-attention mass F  ->  budgeted selection on F
             ->  compaction of the kept K/V rows  ->  one-token decode over the pruned cache

The plan only sequences the C-ABI calls on one stream; it performs no
arithmetic of its own.
"""
from __future__ import annotations

import torch

from . import _lib


class PrefillPrunePlan:
    """Buffers for a [B, H_q, S, D] prefill pruned to per-row budgets (rows = B * H_kv)."""

    def __init__(self, n_batch, h_q, h_kv, seq_len, head_dim, dtype, window, n_sink, n_recent,
                 b_max, device="cuda"):
        self.B, self.Hq, self.Hkv, self.S, self.D = n_batch, h_q, h_kv, seq_len, head_dim
        self.window, self.n_sink, self.n_recent, self.b_max = window, n_sink, n_recent, b_max
        self.dtype = dtype
        R = n_batch * h_kv
        f32, i32 = torch.float32, torch.int32
        self.lse = torch.empty(n_batch, h_q, seq_len, device=device, dtype=f32)
        self.F = torch.empty(n_batch, h_kv, seq_len, device=device, dtype=f32)
        ws = _lib.kvp_future_attn_mass_workspace_size(dtype, n_batch, h_q, h_kv, seq_len, head_dim,
                                                      window)
        self.fam_ws = torch.empty(max(ws, 1), device=device, dtype=torch.uint8)
        self.idx = torch.empty(R, b_max, device=device, dtype=i32)
        self.count = torch.empty(R, device=device, dtype=i32)
        self.kc = torch.zeros(R, b_max, head_dim, device=device, dtype=dtype)
        self.vc = torch.zeros(R, b_max, head_dim, device=device, dtype=dtype)
        self.out = torch.empty(n_batch, h_q, head_dim, device=device, dtype=f32)
        dws = _lib.kvp_decode_attn_workspace_size(n_batch, h_q, h_kv, head_dim, b_max, False)
        self.dec_ws = torch.empty(dws, device=device, dtype=torch.uint8)
        self.launches_per_step = 6   # lse, mass, select, compact, decode split + combine (+ mass reduce)

    def __call__(self, q, k, v, dq, budgets, stream=None):
        R = self.B * self.Hkv
        _lib.kvp_lse_pass(q, k, lse=self.lse, stream=stream)
        _lib.kvp_future_attn_mass(q, k, self.lse, self.window, F=self.F, workspace=self.fam_ws,
                                  stream=stream)
        _lib.kvp_select_topk(self.F.view(R, self.S), budgets, self.n_sink, self.n_recent, self.b_max,
                             idx=self.idx, count=self.count, stream=stream)
        _lib.kvp_compact_kv(k.view(R, self.S, self.D), v.view(R, self.S, self.D), self.idx,
                            self.count, k_out=self.kc, v_out=self.vc, stream=stream)
        _lib.kvp_decode_attn(dq, self.kc, self.vc, self.count, out=self.out, workspace=self.dec_ws,
                             stream=stream)
        return self.out


def prefill_prune_step(q, k, v, dq, budgets, window, n_sink, n_recent, b_max=None):
    """Allocate a plan for these shapes and run one pass (convenience for small calls)."""
    if q.dim() == 3:
        q, k, v, dq = q[None], k[None], v[None], dq[None]
    B, Hq, S, D = q.shape
    b_max = int(budgets.max().item()) if b_max is None else b_max
    b_max = max(b_max, n_sink + n_recent, 1)
    plan = PrefillPrunePlan(B, Hq, k.shape[1], S, D, q.dtype, window, n_sink, n_recent, min(b_max, S),
                            device=q.device)
    plan(q, k, v, dq, budgets)
    return plan
