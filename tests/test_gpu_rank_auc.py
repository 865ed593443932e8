"""GPU parity of row ranking (bit-exact against the oracle's stable ordering) and of the
eviction-cost AUC (1e-9 relative: products and sums in fp64) of KVP's ranking reward, with
F from this library's future-mass pass; and static ranks from scores feeding the cutoffs."""
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


@pytest.mark.parametrize("R,T,mode", [(3, 1, "plain"), (2, 5, "plain"), (3, 4096, "ties"),
                                      (2, 4097, "specials"), (4, 30000, "ties"), (2, 12345, "plain")])
def test_rank_rows_matches_oracle(kvp, R, T, mode):
    s = kvp_inputs.make_scores(R, T, seed=T + R, quantize=4 if mode == "ties" else None,
                               specials=mode == "specials")
    got = kvp.kvp_rank_rows(s.cuda())
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    g = got.cpu().numpy()
    for r in range(R):
        assert (g[r] == oracle.rank_by_scores(s[r].numpy())).all(), f"row {r}"


def test_rank_rows_full_size_and_cutoffs_from_scores(kvp):
    """Qwen3-8B 131k shape: 8 KV heads x 131072 tokens of static scores -> ranks -> cutoffs."""
    w = kvp_inputs.QWEN3_8B_131K
    s = kvp_inputs.make_scores(w.h_kv, w.seq_len, seed=21, device="cuda")
    ranks = kvp.kvp_rank_rows(s)
    k_lr = w.budget - w.n_sink - w.window
    tau = kvp.kvp_topk_cutoffs(ranks, w.n_sink, w.window, k_lr)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    for h in (0, 5):
        want = oracle.rank_by_scores(s[h].cpu().numpy())
        assert (ranks[h].cpu().numpy() == want).all()
        assert (tau[h].cpu().numpy() == oracle.fenwick_cutoffs(want, w.n_sink, w.window, k_lr)).all()


def test_eviction_auc_from_future_mass(kvp):
    w = kvp_inputs.QWEN3_4B_LAYER.scaled(seq_len=700, h_q=8, h_kv=2)
    x = kvp_inputs.make_prefill(w, device="cuda")
    lse = kvp.kvp_lse_pass(x["q"], x["k"])
    F = kvp.kvp_future_attn_mass(x["q"], x["k"], lse, w.window)[0].contiguous()    # [H_kv, S]
    R, T, M = F.shape[0], F.shape[1], 4
    gen = torch.Generator(device="cuda").manual_seed(0)
    rand = torch.stack([torch.stack([torch.randperm(T, generator=gen, device="cuda") for _ in range(M)])
                        for _ in range(R)]).to(torch.int32)
    opt_r = kvp.kvp_rank_rows(F)
    auc = kvp.kvp_eviction_auc(F, rand)
    auc_opt = kvp.kvp_eviction_auc(F, opt_r)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    Fn = F.cpu().numpy().astype(np.float64)
    for r in range(R):
        assert (opt_r[r].cpu().numpy() == oracle.rank_by_scores(F[r].cpu().numpy())).all()
        want_opt = oracle.optimal_auc(Fn[r])
        assert abs(auc_opt[r, 0].item() - want_opt) <= 1e-9 * want_opt
        for m in range(M):
            want = oracle.eviction_auc(Fn[r], rand[r, m].cpu().numpy())
            assert abs(auc[r, m].item() - want) <= 1e-9 * want
            assert auc[r, m].item() >= auc_opt[r, 0].item()


@pytest.mark.parametrize("R,M,T", [(2, 3, 1), (1, 2, 8191), (3, 5, 20003), (2, 4, 16388),
                                   (8, 8, 20003), (4, 16, 16388), (16, 4, 5), (8, 16, 131072)])
def test_eviction_auc_shapes(kvp, R, M, T):
    """Scalar path (T not a multiple of 4), several 8192-entry chunks with a ragged tail, the
    vector path with a 4-entry tail chunk, a single entry, many rankings of short rows, and the
    16-ranking benchmark shape; F spans many binades."""
    gen = torch.Generator(device="cuda").manual_seed(R * 1000 + T)
    F = torch.exp(4.0 * torch.randn(R, T, generator=gen, device="cuda")) * 1e-3
    rk = torch.stack([torch.stack([torch.randperm(T, generator=gen, device="cuda") for _ in range(M)])
                      for _ in range(R)]).to(torch.int32).contiguous()
    auc = kvp.kvp_eviction_auc(F, rk)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    Fn = F.cpu().numpy().astype(np.float64)
    for r in range(R):
        for m in range(M):
            want = oracle.eviction_auc(Fn[r], rk[r, m].cpu().numpy())
            assert abs(auc[r, m].item() - want) <= 1e-9 * want, (r, m, auc[r, m].item(), want)
