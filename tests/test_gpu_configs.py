"""Full-size parity of the two long-context prefill workloads, each run on its own F:

* Qwen3-8B-shaped layer at S = 131072 (32 / 8 heads, w = 256): the row LSE of KV head 3's
  four query heads over every row and F on 2048 strided keys plus the last 2w keys against
  the fp64 oracle (keys near 0 receive mass from all 1024 query tiles, through every chunk of
  the mass pass's partial sums), then selection at b = 16384 (12.5 % retention: 4 sinks, 256
  recent, top-k of F) and compaction of all 8 rows, bit-exact;
* Llama-3.1-8B-shaped 32 layers at S = 32768 (w = 64): per-head budgets from the closed-form
  Soft-TopK at 15 % aggregate retention, selection on the F of all 256 (layer, KV head) rows
  and compaction, bit-exact for every row.

Sources: KVpop, "Defining Future Attention Utility" and Figure 2 (the transposed pass); LKV,
"LKV-H" (b = floor(r * t)); Learning to Evict from Key-Value Cache §4.1 (compaction)."""
import numpy as np
import pytest
import torch

import kvp_inputs
import oracle
from tests.gpu_util import (check_F, check_lse, np64, oracle_future_mass_threads,
                            oracle_row_lse_threads)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvp():
    import learned_kv_cache_gb300 as m
    m.load()
    return m


def _passes(kvp, q, k, window):
    lse = kvp.kvp_lse_pass(q, k)
    F = kvp.kvp_future_attn_mass(q, k, lse, window)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    return lse, F


def _select_compact_exact(kvp, F_rows, budgets, n_sink, n_recent, b_max, k_rows, v_rows):
    """Selection and compaction on the GPU's F, compared bit for bit with the oracle's
    selection of the same F and its gather of the same K / V."""
    b_dev = torch.as_tensor(np.asarray(budgets), dtype=torch.int32, device="cuda")
    idx, count = kvp.kvp_select_topk(F_rows, b_dev, n_sink, n_recent, b_max)
    kc, vc = kvp.kvp_compact_kv(k_rows, v_rows, idx, count)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    idx_r, cnt_r = oracle.select_topk(F_rows.cpu().numpy(), budgets, n_sink, n_recent, b_max=b_max)
    assert np.array_equal(count.cpu().numpy(), cnt_r)
    assert np.array_equal(idx.cpu().numpy(), idx_r)
    R = F_rows.shape[0]
    for r0 in range(0, R, 32):               # bounded host memory: 32 rows at a time
        r1 = min(R, r0 + 32)
        kr, vr = oracle.compact_kv(k_rows[r0:r1].cpu().view(torch.int16).numpy(),
                                   v_rows[r0:r1].cpu().view(torch.int16).numpy(),
                                   idx_r[r0:r1], cnt_r[r0:r1])
        kg = kc[r0:r1].cpu().view(torch.int16).numpy()
        vg = vc[r0:r1].cpu().view(torch.int16).numpy()
        for r in range(r1 - r0):
            n = int(cnt_r[r0 + r])
            assert kg[r, :n].tobytes() == kr[r, :n].tobytes(), r0 + r
            assert vg[r, :n].tobytes() == vr[r, :n].tobytes(), r0 + r
    return idx_r, cnt_r


def test_qwen3_8b_131k_long_rows_and_pipeline(kvp):
    w = kvp_inputs.QWEN3_8B_131K
    x = kvp_inputs.make_prefill(w, device="cuda")
    lse, F = _passes(kvp, x["q"], x["k"], w.window)
    S, G, D = w.seq_len, w.group, w.head_dim
    scale = D ** -0.5
    h = 3
    qs = x["q"][0, h * G:(h + 1) * G].cpu()
    ks = x["k"][0, h:h + 1].cpu()
    lse_r = oracle_row_lse_threads(qs, ks, scale)
    check_lse(np64(lse[0, h * G:(h + 1) * G]), lse_r, "131k every row")
    keys = np.unique(np.concatenate([np.arange(0, S, S // 2048), np.arange(S - 2 * w.window, S)]))
    F_r = oracle_future_mass_threads(qs, ks, lse_r, scale, w.window, keys)
    check_F(np64(F[0, h])[keys][None], F_r, "131k strided keys")
    # 12.5 % retention on the layer's own F: all 8 rows selected and compacted
    R = w.rows
    _, cnt = _select_compact_exact(kvp, F.view(R, S), [w.budget] * R, w.n_sink, w.n_recent, w.budget,
                                   x["k"].view(R, S, D), x["v"].view(R, S, D))
    assert (cnt == w.budget).all()


def test_llama_32_layers_pipeline_on_own_F(kvp):
    w = kvp_inputs.LLAMA31_8B_32L
    x = kvp_inputs.make_prefill(w, device="cuda")
    lse, F = _passes(kvp, x["q"], x["k"], w.window)
    del lse
    R, S, D = w.rows, w.seq_len, w.head_dim
    s = kvp_inputs.make_head_scores(R, w.seed)
    _, b = kvp.kvp_soft_topk_budgets(s.cuda(), w.retention * R, S)
    torch.cuda.synchronize()
    budgets = b.cpu().numpy()
    r_ref, b_ref, _ = oracle.head_budgets(s.numpy(), w.retention, S)
    boundary = np.abs(r_ref * S - np.round(r_ref * S)) < 1e-9     # r*t within 1e-9 of an integer
    assert ((budgets == b_ref) | boundary).all()
    b_max = int(budgets.max())
    _, cnt = _select_compact_exact(kvp, F.view(R, S), budgets, w.n_sink, w.window, b_max,
                                   x["k"].view(R, S, D), x["v"].view(R, S, D))
    assert np.array_equal(cnt, np.maximum(budgets, w.n_sink + w.window))
