"""The whole hot path at the Qwen3-4B-shaped layer size, in the launch configuration the
benchmark times (one PrefillPrunePlan pass), checked stage by stage against the oracle."""
import numpy as np
import pytest
import torch

import kvp_inputs
import oracle
from tests.gpu_util import DECODE_ATOL, check_F, check_lse, np64

pytestmark = pytest.mark.gpu


def test_bench_step_matches_oracle():
    import learned_kv_cache_gb300 as kvp
    from learned_kv_cache_gb300.pipeline import PrefillPrunePlan
    w = kvp_inputs.QWEN3_4B_LAYER
    x = kvp_inputs.make_prefill(w, device="cuda")
    R, S, D, G = w.rows, w.seq_len, w.head_dim, w.group
    plan = PrefillPrunePlan(1, w.h_q, w.h_kv, S, D, x["q"].dtype, w.window, w.n_sink, w.n_recent,
                            w.budget)
    budgets = torch.full((R,), w.budget, dtype=torch.int32, device="cuda")
    for _ in range(2):                      # second pass reuses every buffer
        plan(x["q"], x["k"], x["v"], x["dq"], budgets)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    scale = D ** -0.5
    q, k = x["q"][0].cpu(), x["k"][0].cpu()
    h = 7
    lse_r = oracle.row_lse(q[h * G:(h + 1) * G], k[h:h + 1], scale)
    check_lse(np64(plan.lse[0, h * G:(h + 1) * G]), lse_r, "step lse")
    F_r = oracle.future_attn_mass(q[h * G:(h + 1) * G], k[h:h + 1], lse_r, scale, w.window)
    check_F(np64(plan.F[0, h:h + 1]), F_r, "step F")
    Fg = plan.F.view(R, S).cpu().numpy()
    idx_r, cnt_r = oracle.select_topk(Fg, [w.budget] * R, w.n_sink, w.n_recent, b_max=w.budget)
    assert (plan.idx.cpu().numpy() == idx_r).all() and (plan.count.cpu().numpy() == cnt_r).all()
    k16 = x["k"][0].cpu().view(torch.int16).numpy()
    v16 = x["v"][0].cpu().view(torch.int16).numpy()
    kcr, vcr = oracle.compact_kv(k16, v16, idx_r, cnt_r)
    assert plan.kc.cpu().view(torch.int16).numpy().tobytes() == kcr.tobytes()
    assert plan.vc.cpu().view(torch.int16).numpy().tobytes() == vcr.tobytes()
    kcf = torch.from_numpy(kcr).view(torch.bfloat16)
    vcf = torch.from_numpy(vcr).view(torch.bfloat16)
    ref, _ = oracle.decode_attn(x["dq"].cpu(), kcf, vcf, cnt_r, scale)
    assert np.abs(plan.out.cpu().double().numpy() - ref).max() <= DECODE_ATOL


def test_smoke_entry_point():
    import __graft_entry__
    __graft_entry__.smoke()


def test_host_pipeline_matches_oracle():
    """PrefillPrunePlan.run_from_host (the end-to-end call: pinned host inputs, per-group
    overlapped copies and passes, host outputs) at the Qwen3-4B layer size, twice in a row."""
    from learned_kv_cache_gb300.pipeline import PrefillPrunePlan
    import learned_kv_cache_gb300 as kvp
    w = kvp_inputs.QWEN3_4B_LAYER
    x = kvp_inputs.make_prefill(w)
    R, S, D, G = w.rows, w.seq_len, w.head_dim, w.group
    plan = PrefillPrunePlan(1, w.h_q, w.h_kv, S, D, x["q"].dtype, w.window, w.n_sink, w.n_recent,
                            w.budget)
    budgets = torch.full((R,), w.budget, dtype=torch.int32, device="cuda")
    host = {k: v.pin_memory() for k, v in x.items()}
    out_h = {"F": torch.empty(plan.F.shape, pin_memory=True),
             "idx": torch.empty(plan.idx.shape, dtype=torch.int32, pin_memory=True),
             "count": torch.empty(plan.count.shape, dtype=torch.int32, pin_memory=True),
             "out": torch.empty(plan.out.shape, pin_memory=True)}
    for _ in range(2):
        plan.run_from_host(host["q"], host["k"], host["v"], host["dq"], budgets, out_h)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    scale = D ** -0.5
    q, k = x["q"][0], x["k"][0]
    for h in (0, 5):
        lse_r = oracle.row_lse(q[h * G:(h + 1) * G], k[h:h + 1], scale)
        F_r = oracle.future_attn_mass(q[h * G:(h + 1) * G], k[h:h + 1], lse_r, scale, w.window)
        check_F(out_h["F"][0, h:h + 1].double().numpy(), F_r, f"host pipeline F head {h}")
    Fg = out_h["F"].view(R, S).numpy()
    idx_r, cnt_r = oracle.select_topk(Fg, [w.budget] * R, w.n_sink, w.n_recent, b_max=w.budget)
    assert (out_h["idx"].numpy() == idx_r).all() and (out_h["count"].numpy() == cnt_r).all()
    k16 = x["k"][0].view(torch.int16).numpy()
    v16 = x["v"][0].view(torch.int16).numpy()
    kcr, vcr = oracle.compact_kv(k16, v16, idx_r, cnt_r)
    ref, _ = oracle.decode_attn(x["dq"], torch.from_numpy(kcr).view(torch.bfloat16),
                                torch.from_numpy(vcr).view(torch.bfloat16), cnt_r, scale)
    assert np.abs(out_h["out"].double().numpy() - ref).max() <= DECODE_ATOL
