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
