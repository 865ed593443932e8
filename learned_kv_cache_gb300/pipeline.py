"""One pass of the whole hot path with preallocated device buffers.

prefill K/V  ->  row LSE  ->  future-attention mass F  ->  budgeted selection on F
             ->  compaction of the kept K/V rows  ->  one-token decode over the pruned cache

The plan only sequences the C-ABI calls; it performs no arithmetic of its own.
``PrefillPrunePlan.run_from_host`` runs the same pass from pinned host tensors,
overlapping the host-to-device copies with the passes: the copy stream moves
the KV heads in four slices (each slice's K rows and its query heads); the
LSE pass of a slice starts on the compute stream as soon as the slice has
landed, and its mass pass runs on a second compute stream so that it overlaps
the next slice's LSE pass; V and the decode query follow on the copy stream;
the small outputs come back at the end.
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
        self.device = device
        self._dev_in = None
        self._copy_stream = None
        self._mass_stream = None
        # run_from_host: KV heads per copy slice (they must add up to h_kv); None = four equal slices
        self.kv_slices = None

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

    def run_from_host(self, q_h, k_h, v_h, dq_h, budgets, out_h, stream=None):
        """One pass from pinned host tensors q_h [B,H_q,S,D], k_h/v_h [B,H_kv,S,D], dq_h [B,H_q,D]
        into pinned host outputs out_h = {"F", "idx", "count", "out"} (shapes of the plan's
        buffers).  Everything is enqueued asynchronously; synchronise ``stream`` to read out_h."""
        if self._dev_in is None:
            self._dev_in = {n: torch.empty(t.shape, dtype=t.dtype, device=self.device)
                            for n, t in (("q", q_h), ("k", k_h), ("v", v_h), ("dq", dq_h))}
            self._copy_stream = torch.cuda.Stream(device=self.device)
            self._mass_stream = torch.cuda.Stream(device=self.device)
        d = self._dev_in
        main = torch.cuda.current_stream(self.device) if stream is None else stream
        cs, ms = self._copy_stream, self._mass_stream
        cs.wait_stream(main)                      # the previous pass is done with the buffers
        ms.wait_stream(main)
        B, Hq, Hkv, S, D = self.B, self.Hq, self.Hkv, self.S, self.D
        G = Hq // Hkv
        R = B * Hkv
        if self.kv_slices is None:
            gs = max(1, Hkv // 4)                 # KV heads per slice
            widths = [min(gs, Hkv - h0) for h0 in range(0, Hkv, gs)]
        else:
            widths = [int(x) for x in self.kv_slices]
            if sum(widths) != Hkv or min(widths) < 1:
                raise ValueError(f"kv_slices {widths} must be positive and add up to h_kv = {Hkv}")
        bounds = [sum(widths[:i]) for i in range(len(widths) + 1)]
        slices = [(b, bounds[i], bounds[i + 1]) for b in range(B) for i in range(len(widths))]
        ready = []
        with torch.cuda.stream(cs):
            for b, h0, h1 in slices:
                d["k"][b, h0:h1].copy_(k_h[b, h0:h1], non_blocking=True)
                d["q"][b, h0 * G:h1 * G].copy_(q_h[b, h0 * G:h1 * G], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cs)
                ready.append(ev)
            d["v"].copy_(v_h, non_blocking=True)
            d["dq"].copy_(dq_h, non_blocking=True)
            v_ready = torch.cuda.Event()
            v_ready.record(cs)
        for (b, h0, h1), ev in zip(slices, ready):
            main.wait_event(ev)
            qg = d["q"][b, h0 * G:h1 * G][None]
            kg = d["k"][b, h0:h1][None]
            lse_g = self.lse[b, h0 * G:h1 * G][None]
            _lib.kvp_lse_pass(qg, kg, lse=lse_g, stream=main)
            lse_done = torch.cuda.Event()
            lse_done.record(main)
            ms.wait_event(lse_done)
            _lib.kvp_future_attn_mass(qg, kg, lse_g, self.window, F=self.F[b, h0:h1][None],
                                      workspace=self.fam_ws, stream=ms)
        mass_done = torch.cuda.Event()
        mass_done.record(ms)
        main.wait_event(mass_done)
        _lib.kvp_select_topk(self.F.view(R, S), budgets, self.n_sink, self.n_recent, self.b_max,
                             idx=self.idx, count=self.count, stream=main)
        main.wait_event(v_ready)
        _lib.kvp_compact_kv(d["k"].view(R, S, D), d["v"].view(R, S, D), self.idx, self.count,
                            k_out=self.kc, v_out=self.vc, stream=main)
        _lib.kvp_decode_attn(d["dq"], self.kc, self.vc, self.count, out=self.out, workspace=self.dec_ws,
                             stream=main)
        with torch.cuda.stream(main):
            out_h["F"].copy_(self.F, non_blocking=True)
            out_h["idx"].copy_(self.idx, non_blocking=True)
            out_h["count"].copy_(self.count, non_blocking=True)
            out_h["out"].copy_(self.out, non_blocking=True)
        return out_h


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
