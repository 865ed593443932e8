"""GPU parity of selection, compaction and the Soft-TopK budgets (bit-exact where integer)."""
import numpy as np
import pytest
import torch

import kvp_inputs
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvp():
    import learned_kv_cache_gb300 as m
    m.load()
    return m


def _select(kvp, scores, budgets, n_sink, n_recent, b_max):
    s = scores.cuda()
    b = torch.as_tensor(np.asarray(budgets), dtype=torch.int32).cuda()
    idx, count = kvp.kvp_select_topk(s, b, n_sink, n_recent, b_max)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    idx_r, cnt_r = oracle.select_topk(scores.numpy(), budgets, n_sink, n_recent, b_max=b_max)
    assert (count.cpu().numpy() == cnt_r).all()
    assert (idx.cpu().numpy() == idx_r).all()
    return idx, count


@pytest.mark.parametrize("R,T,quant,specials", [(1, 256, None, False), (8, 8192, None, False),
                                                (5, 3001, 4, False), (3, 20000, 2, True),
                                                (2, 131072, None, True), (4, 100, 1, True)])
def test_select_matches_oracle(kvp, R, T, quant, specials):
    scores = kvp_inputs.make_scores(R, T, seed=T + R, quantize=quant, specials=specials)
    n_sink, n_recent = 4, min(128, T // 8)
    rng = np.random.default_rng(T)
    budgets = rng.integers(0, T + 10, size=R)
    budgets[0] = n_sink + n_recent          # k = 0
    b_max = int(max(budgets.max(), n_sink + n_recent))
    b_max = min(b_max, T)
    _select(kvp, scores, budgets, n_sink, n_recent, b_max)


def test_select_all_equal_scores_takes_lowest_indices(kvp):
    scores = torch.zeros(3, 5000)
    idx, count = _select(kvp, scores, [100, 1000, 4999], 4, 16, 4999)
    assert idx[0, :100].cpu().tolist() == list(range(84)) + list(range(4984, 5000))


def test_select_nested_across_budgets(kvp):
    scores = kvp_inputs.make_scores(1, 4096, seed=9, quantize=8)
    prev = set()
    for b in range(64, 4097, 257):
        idx, count = _select(kvp, scores, [b], 4, 32, 4096)
        cur = set(idx[0, :int(count[0])].cpu().tolist())
        assert prev <= cur
        prev = cur


def test_select_reports_budget_overflow(kvp):
    s = torch.randn(2, 100).cuda()
    b = torch.tensor([50, 90], dtype=torch.int32).cuda()
    idx, count = kvp.kvp_select_topk(s, b, 2, 2, 60)
    with pytest.raises(kvp.KvpError) as e:
        kvp.kvp_check_device_status()
    assert e.value.status == -6
    assert count.cpu().tolist() == [50, -1]
    kvp.kvp_check_device_status()     # cleared by the read


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f16", 128), ("f32", 64), ("bf16", 64)])
def test_compact_bit_exact(kvp, dtype, D):
    R, T = 6, 3000
    gen = torch.Generator().manual_seed(D)
    dt = kvp_inputs.torch_dtype(dtype)
    k = torch.randn(R, T, D, generator=gen).to(dt)
    v = torch.randn(R, T, D, generator=gen).to(dt)
    scores = kvp_inputs.make_scores(R, T, seed=3)
    budgets = [500, 64, 3000, 1, 2999, 777]
    idx, count = _select(kvp, scores, budgets, 4, 32, 3000)
    kc, vc = kvp.kvp_compact_kv(k.cuda(), v.cuda(), idx, count)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    idx_r, cnt_r = oracle.select_topk(scores.numpy(), budgets, 4, 32, b_max=3000)
    kr, vr = oracle.compact_kv(k.view(torch.int16 if dt != torch.float32 else torch.int32).numpy(),
                               v.view(torch.int16 if dt != torch.float32 else torch.int32).numpy(),
                               idx_r, cnt_r)
    kg = kc.cpu().view(torch.int16 if dt != torch.float32 else torch.int32).numpy()
    vg = vc.cpu().view(torch.int16 if dt != torch.float32 else torch.int32).numpy()
    for r in range(R):
        n = int(cnt_r[r])
        assert kg[r, :n].tobytes() == kr[r, :n].tobytes()
        assert vg[r, :n].tobytes() == vr[r, :n].tobytes()


def test_compact_reports_bad_index(kvp):
    k = torch.zeros(1, 10, 128, dtype=torch.bfloat16).cuda()
    idx = torch.tensor([[0, 3, 10, -1]], dtype=torch.int32).cuda()
    count = torch.tensor([3], dtype=torch.int32).cuda()
    kvp.kvp_compact_kv(k, k, idx, count)
    with pytest.raises(kvp.KvpError):
        kvp.kvp_check_device_status()


@pytest.mark.parametrize("n,retention,t,seed", [(256, 0.15, 32768, 2), (1024, 0.3, 1000, 5),
                                                (7, 0.5, 100, 1), (1, 0.5, 10, 0)])
def test_soft_topk_budgets(kvp, n, retention, t, seed):
    s = kvp_inputs.make_head_scores(n, seed)
    r_g, b_g = kvp.kvp_soft_topk_budgets(s.cuda(), retention * n, t)
    torch.cuda.synchronize()
    r_r, b_r, _ = oracle.head_budgets(s.numpy(), retention, t)
    r_g = r_g.cpu().numpy()
    np.testing.assert_allclose(r_g, r_r, rtol=1e-12, atol=0)
    b_g = b_g.cpu().numpy()
    boundary = np.abs(r_r * t - np.round(r_r * t)) < 1e-9
    assert ((b_g == b_r) | boundary).all()


def test_llama_budgets_select_compact_all_rows(kvp):
    """Llama-3.1-8B recipe: 256 head budgets from the Soft-TopK at 15 % retention, then
    selection and compaction of all 256 rows (T = 32768) on seeded scores."""
    w = kvp_inputs.LLAMA31_8B_32L
    s = kvp_inputs.make_head_scores(w.rows, w.seed)
    _, b = kvp.kvp_soft_topk_budgets(s.cuda(), w.retention * w.rows, w.seq_len)
    budgets = b.cpu().numpy()
    b_max = int(budgets.max())
    scores = kvp_inputs.make_scores(w.rows, w.seq_len, seed=11)
    idx, count = _select(kvp, scores, budgets, w.n_sink, w.window, b_max)
    gen = torch.Generator(device="cuda").manual_seed(1)
    k = torch.randn(w.rows, w.seq_len, 128, generator=gen, device="cuda").to(torch.bfloat16)
    v = torch.randn(w.rows, w.seq_len, 128, generator=gen, device="cuda").to(torch.bfloat16)
    kc, vc = kvp.kvp_compact_kv(k, v, idx, count)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    for r in (0, 100, 255):
        idx_r, cnt_r = oracle.select_topk(scores[r:r + 1].numpy(), budgets[r:r + 1], w.n_sink,
                                          w.window, b_max=b_max)
        kr, vr = oracle.compact_kv(k[r:r + 1].cpu().view(torch.int16).numpy(),
                                   v[r:r + 1].cpu().view(torch.int16).numpy(), idx_r, cnt_r)
        n = int(cnt_r[0])
        assert kc[r, :n].cpu().view(torch.int16).numpy().tobytes() == kr[0, :n].tobytes()
        assert vc[r, :n].cpu().view(torch.int16).numpy().tobytes() == vr[0, :n].tobytes()
