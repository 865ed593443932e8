"""GPU parity of KVpop's running top-k cutoffs (bit-exact against the oracle's Fenwick tree)
and of the sparse row LSE under that mask (fp32 path: 1e-3 absolute, as the dense LSE), and of
the future-attention mass computed from the sparse LSE (2e-3 relative, as F)."""
import numpy as np
import pytest
import torch

import kvp_inputs
import oracle
from tests.gpu_util import check_F, check_lse, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvp():
    import learned_kv_cache_gb300 as m
    m.load()
    return m


@pytest.mark.parametrize("H,S,s,w,k", [
    (3, 1, 0, 0, 1), (2, 100, 4, 16, 8), (2, 1000, 4, 64, 37), (1, 1537, 0, 0, 1),
    (2, 3000, 4, 128, 700), (1, 2048, 2, 5000, 3), (1, 700, 4, 16, 5000), (4, 5001, 4, 64, 1200),
    (2, 16384, 4, 128, 3000), (1, 20000, 4, 128, 4000), (1, 70001, 4, 128, 9000),
])
def test_cutoffs_match_fenwick_oracle(kvp, H, S, s, w, k):
    ranks = kvp_inputs.make_static_ranks(H, S, seed=S + k)
    tau = kvp.kvp_topk_cutoffs(ranks.cuda(), s, w, k)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    got = tau.cpu().numpy()
    for h in range(H):
        want = oracle.fenwick_cutoffs(ranks[h].numpy(), s, w, k)
        assert (got[h] == want).all(), f"head {h}: first diff at {np.argmax(got[h] != want)}"


def test_cutoffs_flag_repeated_ranks(kvp):
    ranks = kvp_inputs.make_static_ranks(1, 600, seed=1)
    ranks[0, 100] = ranks[0, 50]
    kvp.kvp_topk_cutoffs(ranks.cuda(), 0, 4, 10)
    with pytest.raises(kvp.KvpError):
        kvp.kvp_check_device_status()
    with pytest.raises(kvp.KvpError):
        kvp.kvp_topk_cutoffs(ranks.cuda(), 0, 4, 0)


def _sparse_case(kvp, dtype, D, S, Hq, Hkv, s, w, k, seed):
    gen = torch.Generator().manual_seed(seed)
    dt = kvp_inputs.torch_dtype(dtype)
    q = (torch.randn(1, Hq, S, D, generator=gen) * 1.5).to(dt)
    kk = torch.randn(1, Hkv, S, D, generator=gen).to(dt)
    ranks = kvp_inputs.make_static_ranks(Hkv, S, seed=seed)
    tau = kvp.kvp_topk_cutoffs(ranks.cuda(), s, w, k)
    lse = kvp.kvp_sparse_lse_pass(q.cuda(), kk.cuda(), ranks.cuda(), tau, s, w)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    return q, kk, ranks, tau.cpu().numpy(), lse


@pytest.mark.parametrize("dtype,D,S,Hq,Hkv,s,w,k", [
    ("bf16", 128, 1000, 4, 2, 4, 64, 100),     # tensor-core path, ranks rows 16-byte aligned
    ("f16", 128, 777, 2, 1, 3, 17, 50),        # tensor-core path, scalar rank loads
    ("bf16", 128, 300, 2, 2, 0, 0, 1),         # window 0, one kept eligible key per query
    ("f32", 64, 513, 4, 2, 4, 16, 40),         # fp32 FFMA path
    ("bf16", 64, 400, 2, 1, 2, 8, 3000),       # k never reached: every eligible key kept
])
def test_sparse_lse_matches_oracle(kvp, dtype, D, S, Hq, Hkv, s, w, k):
    q, kk, ranks, tau, lse = _sparse_case(kvp, dtype, D, S, Hq, Hkv, s, w, k, seed=S + D)
    want = oracle.sparse_row_lse(q[0], kk[0], ranks.numpy(), tau, D ** -0.5, s, w)
    check_lse(np64(lse[0]), want, f"{dtype} D{D} S{S}")
    if k >= S:
        dense = oracle.row_lse(q[0], kk[0], D ** -0.5)
        assert np.abs(np64(lse[0]) - dense).max() < 1e-3


@pytest.mark.parametrize("dtype,D,scale", [
    ("bf16", 128, None),     # rank-ordered tiles mask out-of-range keys in the contraction
    ("f16", 128, None),
    ("f16", 64, None),
    ("bf16", 128, 1e-4),     # a small scale: the masking step's factors are still bf16 normals
    ("f16", 128, 1e-4),      # 2^a * 2^b out of f16's range: every key's position tested instead
])
def test_sparse_lse_rank_ordered_stream(kvp, dtype, D, scale):
    """A small long-range budget (k = 80 of 3000) so most query tiles take the rank-ordered
    stream.  Keys planted after a query with a large logit for it (a multiple of that query)
    are ranked first, so they sit in the first rank-ordered tiles of every earlier query tile,
    where only the mask removes them: a missed key adds e^(~100) to its row."""
    S, Hq, Hkv, s, w, k = 3000, 4, 2, 4, 64, 80
    gen = torch.Generator().manual_seed(D + (0 if scale is None else 1))
    dt = kvp_inputs.torch_dtype(dtype)
    q = torch.randn(1, Hq, S, D, generator=gen)
    kk = torch.randn(1, Hkv, S, D, generator=gen)
    G = Hq // Hkv
    planted = torch.randint(1500, S, (Hkv, 6), generator=gen)
    for h in range(Hkv):
        for j in planted[h].tolist():
            kk[0, h, j] = q[0, h * G, j - 600] * 2.0
    q, kk = q.to(dt), kk.to(dt)
    ranks = kvp_inputs.make_static_ranks(Hkv, S, seed=D)
    for h in range(Hkv):                        # planted keys take the smallest ranks
        pl = planted[h].unique()
        rest = torch.ones(S, dtype=torch.bool)
        rest[pl] = False
        order = ranks[h].argsort()
        order = order[rest[order]]              # the other keys keep their relative order
        ranks[h, pl] = torch.arange(len(pl), dtype=ranks.dtype)
        ranks[h, order] = torch.arange(len(pl), S, dtype=ranks.dtype)
    sc = D ** -0.5 if scale is None else scale
    tau = kvp.kvp_topk_cutoffs(ranks.cuda(), s, w, k)
    lse = kvp.kvp_sparse_lse_pass(q.cuda(), kk.cuda(), ranks.cuda(), tau, s, w, sm_scale=sc)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    want = oracle.sparse_row_lse(q[0], kk[0], ranks.numpy(), tau.cpu().numpy(), sc, s, w)
    check_lse(np64(lse[0]), want, f"{dtype} D{D} scale {scale}")


def test_future_mass_from_sparse_lse(kvp):
    dtype, D, S, Hq, Hkv, s, w, k = "bf16", 128, 900, 4, 2, 4, 32, 200
    q, kk, ranks, tau, lse = _sparse_case(kvp, dtype, D, S, Hq, Hkv, s, w, k, seed=11)
    F = kvp.kvp_future_attn_mass(q.cuda(), kk.cuda(), lse, w)
    torch.cuda.synchronize()
    sl = oracle.sparse_row_lse(q[0], kk[0], ranks.numpy(), tau, D ** -0.5, s, w)
    want = oracle.future_attn_mass(q[0], kk[0], sl, D ** -0.5, w)
    check_F(np64(F[0]), want, "F from the sparse LSE")


def test_sparse_lse_qwen3_4b_layer_full_size(kvp):
    """S = 8192, 32/8 heads, long-range budget k = budget - sinks - window; KV head 5's four
    query heads checked on 192 sampled rows plus the last 64."""
    w = kvp_inputs.QWEN3_4B_LAYER
    x = kvp_inputs.make_prefill(w, device="cuda")
    k_lr = w.budget - w.n_sink - w.window
    ranks = kvp_inputs.make_static_ranks(w.h_kv, w.seq_len, seed=3, device="cuda")
    tau = kvp.kvp_topk_cutoffs(ranks, w.n_sink, w.window, k_lr)
    lse = kvp.kvp_sparse_lse_pass(x["q"], x["k"], ranks, tau, w.n_sink, w.window)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    h, G = 5, w.group
    rows = np.unique(np.concatenate([np.random.default_rng(0).integers(0, w.seq_len, 192),
                                     np.arange(w.seq_len - 64, w.seq_len)]))
    want_tau = oracle.fenwick_cutoffs(ranks[h].cpu().numpy(), w.n_sink, w.window, k_lr)
    assert (tau[h].cpu().numpy() == want_tau).all()
    want = oracle.sparse_row_lse(x["q"][0, h * G:(h + 1) * G].cpu(), x["k"][0, h:h + 1].cpu(),
                                 ranks[h:h + 1].cpu().numpy(), want_tau[None], w.head_dim ** -0.5,
                                 w.n_sink, w.window, rows=rows)
    check_lse(np64(lse[0, h * G:(h + 1) * G])[:, rows], want, "full-size sparse LSE")


@pytest.mark.parametrize("S", [1, 77, 129])
def test_sparse_lse_short_sequences(kvp, S):
    """A single (partial) tile, S below the window, and one full tile plus one key."""
    q, kk, ranks, tau, lse = _sparse_case(kvp, "bf16", 128, S, 4, 2, 2, 16, 5, seed=S)
    want = oracle.sparse_row_lse(q[0], kk[0], ranks.numpy(), tau, 128 ** -0.5, 2, 16)
    check_lse(np64(lse[0]), want, f"S{S}")


def test_sparse_lse_qwen3_8b_131k_sampled(kvp):
    """131072 tokens, one KV head: cutoffs in full, the sparse LSE on 96 sampled rows."""
    w = kvp_inputs.QWEN3_8B_131K
    x = kvp_inputs.make_prefill_layer(w, 0, device="cuda", seq_len=w.seq_len)
    q = x["q"][None, :w.group].contiguous()          # KV head 0 and its query heads
    k = x["k"][None, :1].contiguous()
    k_lr = w.budget - w.n_sink - w.window
    ranks = kvp_inputs.make_static_ranks(1, w.seq_len, seed=9, device="cuda")
    tau = kvp.kvp_topk_cutoffs(ranks, w.n_sink, w.window, k_lr)
    lse = kvp.kvp_sparse_lse_pass(q, k, ranks, tau, w.n_sink, w.window)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    want_tau = oracle.fenwick_cutoffs(ranks[0].cpu().numpy(), w.n_sink, w.window, k_lr)
    assert (tau[0].cpu().numpy() == want_tau).all()
    rows = np.unique(np.concatenate([np.random.default_rng(1).integers(0, w.seq_len, 80),
                                     np.arange(w.seq_len - 16, w.seq_len)]))
    want = oracle.sparse_row_lse(q[0].cpu(), k[0].cpu(), ranks.cpu().numpy(), want_tau[None],
                                 w.head_dim ** -0.5, w.n_sink, w.window, rows=rows)
    check_lse(np64(lse[0])[:, rows], want, "131k sparse LSE")


def test_sparse_lse_any_cutoffs_and_ranks(kvp):
    """The mask is applied as written: cutoffs that are not monotone (drawn at random) with valid
    ranks (the rank-ordered stream must cover every row's cutoff), and ranks that are not a
    permutation (the pass falls back to the dense stream)."""
    S, Hq, Hkv, D, s, w = 1024, 4, 2, 128, 4, 32
    gen = torch.Generator().manual_seed(77)
    q = torch.randn(1, Hq, S, D, generator=gen).to(torch.bfloat16)
    kk = torch.randn(1, Hkv, S, D, generator=gen).to(torch.bfloat16)
    ranks = kvp_inputs.make_static_ranks(Hkv, S, seed=5)
    tau = torch.randint(100, 400, (Hkv, S), generator=gen).to(torch.int32)
    tau[:, :200] = -1
    lse = kvp.kvp_sparse_lse_pass(q.cuda(), kk.cuda(), ranks.cuda(), tau.cuda(), s, w)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    want = oracle.sparse_row_lse(q[0], kk[0], ranks.numpy(), tau.numpy(), D ** -0.5, s, w)
    check_lse(np64(lse[0]), want, "random cutoffs")
    bad = ranks.clone()
    bad[0, 10] = bad[0, 20]                      # not a permutation
    tau2 = torch.full((Hkv, S), 300, dtype=torch.int32)
    lse2 = kvp.kvp_sparse_lse_pass(q.cuda(), kk.cuda(), bad.cuda(), tau2.cuda(), s, w)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    want2 = oracle.sparse_row_lse(q[0], kk[0], bad.numpy(), tau2.numpy(), D ** -0.5, s, w)
    check_lse(np64(lse2[0]), want2, "ranks not a permutation")
