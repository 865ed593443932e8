"""GPU parity of single-token decode attention (with the optional key mass)."""
import numpy as np
import pytest
import torch

import kvp_inputs
import oracle
from tests.gpu_util import DECODE_ATOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvp():
    import learned_kv_cache_gb300 as m
    m.load()
    return m


def _mass_close(got, want):
    got = np.asarray(got, np.float64)
    assert (np.abs(got - want) <= 2e-3 * np.abs(want) + 1e-9).all(), np.abs(got - want).max()


@pytest.mark.parametrize("dtype,D,G", [("f16", 128, 6), ("bf16", 128, 4), ("f32", 64, 2),
                                       ("bf16", 64, 8), ("f32", 128, 1), ("f16", 64, 3)])
def test_decode_ragged_lengths(kvp, dtype, D, G):
    L, Hkv, T_cap = 3, 2, 1500
    R = L * Hkv
    dt = kvp_inputs.torch_dtype(dtype)
    gen = torch.Generator().manual_seed(D * 10 + G)
    q = torch.randn(L, G * Hkv, D, generator=gen).to(dt)
    kc = (torch.randn(R, T_cap, D, generator=gen) * 2).to(dt)
    vc = torch.randn(R, T_cap, D, generator=gen).to(dt)
    lens = torch.tensor([1500, 1, 0, 777, 64, 1499], dtype=torch.int32)
    mass = torch.full((R, T_cap), 7.0, device="cuda")
    out = kvp.kvp_decode_attn(q.cuda(), kc.cuda(), vc.cuda(), lens.cuda(), key_mass=mass)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    ref, mref = oracle.decode_attn(q, kc, vc, lens.numpy(), D ** -0.5)
    err = np.abs(out.cpu().double().numpy() - ref).max()
    assert err <= DECODE_ATOL, err
    _mass_close(mass.cpu().numpy(), mref)
    # accumulate = 1 adds a second helping
    kvp.kvp_decode_attn(q.cuda(), kc.cuda(), vc.cuda(), lens.cuda(), key_mass=mass, accumulate=True)
    torch.cuda.synchronize()
    _mass_close(mass.cpu().numpy(), 2 * mref)


@pytest.mark.parametrize("L,Hkv,T_cap,use_pos", [
    (6, 2, 3000, False),     # rows split over a cluster of CTAs, logits in shared memory
    (20, 2, 12000, True),    # cluster, more keys per CTA than shared memory holds: workspace logits
    (1, 2, 20000, True),     # more than 8 CTAs per row: partials merged by the last CTA, second pass
])
def test_decode_key_mass_paths(kvp, L, Hkv, T_cap, use_pos):
    """The key mass through each way the decode kernel can form it, with ragged lengths,
    optional source positions and accumulation."""
    G, D = 4, 128
    R = L * Hkv
    gen = torch.Generator().manual_seed(T_cap + R)
    q = torch.randn(L, G * Hkv, D, generator=gen).to(torch.bfloat16)
    kc = (torch.randn(R, T_cap, D, generator=gen) * 1.5).to(torch.bfloat16)
    vc = torch.randn(R, T_cap, D, generator=gen).to(torch.bfloat16)
    lens = torch.randint(T_cap // 2, T_cap + 1, (R,), generator=gen).to(torch.int32)
    lens[0] = T_cap
    T_src = T_cap * 2 if use_pos else T_cap
    pos = None
    if use_pos:
        pos = torch.stack([torch.randperm(T_src, generator=gen)[:T_cap].sort().values
                           for _ in range(R)]).to(torch.int32)
    mass = torch.full((R, T_src), 3.0, device="cuda")
    out = kvp.kvp_decode_attn(q.cuda(), kc.cuda(), vc.cuda(), lens.cuda(), key_mass=mass,
                              key_pos=None if pos is None else pos.cuda())
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    ref, mref = oracle.decode_attn(q, kc, vc, lens.numpy(), D ** -0.5,
                                   key_pos=None if pos is None else pos.numpy(), T_src=T_src)
    assert np.abs(out.cpu().double().numpy() - ref).max() <= DECODE_ATOL
    _mass_close(mass.cpu().numpy(), mref)
    kvp.kvp_decode_attn(q.cuda(), kc.cuda(), vc.cuda(), lens.cuda(), key_mass=mass,
                        key_pos=None if pos is None else pos.cuda(), accumulate=True)
    torch.cuda.synchronize()
    _mass_close(mass.cpu().numpy(), 2 * mref)


def test_decode_single_key_and_identical_keys(kvp):
    D = 128
    v = torch.randn(2, 64, D).to(torch.bfloat16)
    k = torch.randn(2, 1, D).to(torch.bfloat16).expand(2, 64, D).contiguous()
    q = torch.randn(1, 4, D).to(torch.bfloat16)
    out = kvp.kvp_decode_attn(q.cuda(), k.cuda(), v.cuda(), torch.tensor([1, 64], dtype=torch.int32).cuda())
    torch.cuda.synchronize()
    o = out.cpu().double()
    assert torch.allclose(o[0, :2], v[0, 0].double().expand(2, D), atol=1e-6)
    assert torch.allclose(o[0, 2:], v[1].double().mean(0).expand(2, D), atol=1e-5)


def test_decode_with_key_positions_scatter(kvp):
    """key_pos maps retained slots to source positions of a T_src-long history."""
    R, T_cap, T_src, D = 2, 40, 1000, 128
    q = torch.randn(1, 4, D).to(torch.float16)
    kc = torch.randn(R, T_cap, D).to(torch.float16)
    vc = torch.randn(R, T_cap, D).to(torch.float16)
    pos = torch.stack([torch.randperm(T_src)[:T_cap].sort().values for _ in range(R)]).to(torch.int32)
    lens = torch.tensor([40, 17], dtype=torch.int32)
    mass = torch.zeros(R, T_src, device="cuda")
    kvp.kvp_decode_attn(q.cuda(), kc.cuda(), vc.cuda(), lens.cuda(), key_mass=mass,
                        key_pos=pos.cuda())
    torch.cuda.synchronize()
    _, mref = oracle.decode_attn(q, kc, vc, lens.numpy(), D ** -0.5, key_pos=pos.numpy(), T_src=T_src)
    _mass_close(mass.cpu().numpy(), mref)


def test_decode_rejects_bad_length(kvp):
    q = torch.randn(1, 2, 128).to(torch.bfloat16).cuda()
    kc = torch.randn(1, 16, 128).to(torch.bfloat16).cuda()
    kvp.kvp_decode_attn(q, kc, kc, torch.tensor([17], dtype=torch.int32).cuda())
    with pytest.raises(kvp.KvpError):
        kvp.kvp_check_device_status()


@pytest.fixture(scope="module")
def qwen25_cache():
    return kvp_inputs.make_decode_cache(kvp_inputs.QWEN25_15B_DECODE, device="cuda")


@pytest.mark.parametrize("budget", list(kvp_inputs.QWEN25_15B_DECODE.decode_budgets))
def test_qwen25_decode_eviction_full_size(kvp, qwen25_cache, budget):
    """Qwen2.5-1.5B-shaped decode eviction at T = 120000 (28 layers, 12/2 heads, fp16), at each
    of the blog's budgets 512 / 1024 / 2048 / 4096: control decode over the full cache with key
    mass, selection on that mass (4 sinks, 32 recent), compaction, pruned decode; selection of
    all 56 rows bit-exact, the rest checked per layer against the oracle."""
    w = kvp_inputs.QWEN25_15B_DECODE
    x = qwen25_cache
    R, T, D = w.rows, w.seq_len, w.head_dim
    full_len = torch.full((R,), T, dtype=torch.int32, device="cuda")
    mass = torch.empty(R, T, device="cuda")
    out_full = kvp.kvp_decode_attn(x["q"], x["k"], x["v"], full_len, key_mass=mass)
    budgets = torch.full((R,), budget, dtype=torch.int32, device="cuda")
    idx, count = kvp.kvp_select_topk(mass, budgets, w.n_sink, w.n_recent, budget)
    kc, vc = kvp.kvp_compact_kv(x["k"], x["v"], idx, count)
    out = kvp.kvp_decode_attn(x["q"], kc, vc, count)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    mass_h = mass.cpu().numpy()
    idx_r, cnt_r = oracle.select_topk(mass_h, [budget] * R, w.n_sink, w.n_recent, b_max=budget)
    assert (idx.cpu().numpy() == idx_r).all() and (count.cpu().numpy() == cnt_r).all()
    scale = D ** -0.5
    for layer in (0, 13, 27):
        rows = slice(layer * w.h_kv, (layer + 1) * w.h_kv)
        kl = x["k"][rows].cpu()
        vl = x["v"][rows].cpu()
        ql = x["q"][layer:layer + 1].cpu()
        ref_full, mref = oracle.decode_attn(ql, kl, vl, [T] * w.h_kv, scale)
        assert np.abs(out_full[layer].cpu().double().numpy() - ref_full[0]).max() <= DECODE_ATOL
        _mass_close(mass_h[rows], mref)
        kcr, vcr = oracle.compact_kv(kl.view(torch.int16).numpy(), vl.view(torch.int16).numpy(),
                                     idx_r[rows], cnt_r[rows])
        assert kc[rows].cpu().view(torch.int16).numpy().tobytes() == kcr.tobytes()
        assert vc[rows].cpu().view(torch.int16).numpy().tobytes() == vcr.tobytes()
        ref, _ = oracle.decode_attn(ql, kcr.view(np.float16), vcr.view(np.float16), cnt_r[rows], scale)
        assert np.abs(out[layer].cpu().double().numpy() - ref[0]).max() <= DECODE_ATOL
