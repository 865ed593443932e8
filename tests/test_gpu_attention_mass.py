"""GPU parity of the row-LSE and future-attention-mass passes against the fp64 oracle."""
import math

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


def _run(kvp, q, k, window, scale=None):
    lse = kvp.kvp_lse_pass(q, k, sm_scale=scale)
    F = kvp.kvp_future_attn_mass(q, k, lse, window, sm_scale=scale)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    return lse, F


def _oracle(q, k, window, scale, rows=None, keys=None):
    lse = oracle.row_lse(q, k, scale)
    F = oracle.future_attn_mass(q, k, lse, scale, window, keys=keys)
    return lse, F


def test_tiny_workload_full(kvp):
    w = kvp_inputs.TINY
    x = kvp_inputs.make_prefill(w)
    scale = w.head_dim ** -0.5
    lse, F = _run(kvp, x["q"].cuda(), x["k"].cuda(), w.window)
    lse_r, F_r = _oracle(x["q"][0], x["k"][0], w.window, scale)
    check_lse(np64(lse[0]), lse_r, "tiny")
    check_F(np64(F[0]), F_r, "tiny")


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("D", [64, 128])
def test_reduced_qwen3_recipe(kvp, dtype, D):
    """Qwen3-4B recipe (sinks, retrieval keys, per-head key scales) at S = 1000: several
    tiles of every size used plus a ragged tail."""
    w = kvp_inputs.QWEN3_4B_LAYER.scaled(seq_len=1000, head_dim=D, dtype=dtype, h_q=8, h_kv=2)
    x = kvp_inputs.make_prefill(w)
    scale = D ** -0.5
    lse, F = _run(kvp, x["q"].cuda(), x["k"].cuda(), w.window)
    lse_r, F_r = _oracle(x["q"][0], x["k"][0], w.window, scale)
    check_lse(np64(lse[0]), lse_r, f"{dtype} D{D}")
    check_F(np64(F[0]), F_r, f"{dtype} D{D}")


@pytest.mark.parametrize("S,w,Hq,Hkv,B", [(1, 0, 2, 1, 1), (2, 0, 1, 1, 1), (129, 0, 4, 1, 1),
                                          (300, 299, 2, 2, 1), (77, 100, 3, 1, 1),
                                          (513, 7, 8, 8, 2), (256, 128, 6, 2, 3)])
def test_edge_shapes(kvp, S, w, Hq, Hkv, B):
    """S = 1, w = 0 (diagonal included), w = S-1, w >= S (everything 0), G = 1,
    several independent problems (n_batch)."""
    gen = torch.Generator().manual_seed(S * 31 + w)
    q = torch.randn(B, Hq, S, 128, generator=gen).to(torch.bfloat16)
    k = torch.randn(B, Hkv, S, 128, generator=gen).to(torch.bfloat16)
    scale = 128 ** -0.5
    lse, F = _run(kvp, q.cuda(), k.cuda(), w)
    for b in range(B):
        lse_r, F_r = _oracle(q[b], k[b], w, scale)
        check_lse(np64(lse[b]), lse_r, f"edge S{S} w{w} b{b}")
        check_F(np64(F[b]), F_r, f"edge S{S} w{w} b{b}")


def test_uniform_attention_closed_form_on_gpu(kvp):
    """K = 0: lse_i = ln(i+1) and F[j] = G (H_S - H_{j+w}) exactly representable inputs."""
    S, w, G = 700, 50, 4
    q = torch.randn(G, S, 128).to(torch.bfloat16).cuda()
    k = torch.zeros(1, S, 128, dtype=torch.bfloat16).cuda()
    lse, F = _run(kvp, q, k, w)
    check_lse(np64(lse), np.log(np.arange(1, S + 1))[None].repeat(G, 0), "uniform")
    H = np.concatenate([[0.0], np.cumsum(1.0 / np.arange(1, S + 1))])
    want = np.array([G * (H[S] - H[j + w]) if j <= S - 1 - w else 0.0 for j in range(S)])
    check_F(np64(F), want[None], "uniform")


def test_qwen3_4b_layer_full_size(kvp):
    """Full Qwen3-4B-shaped layer (S = 8192, 32/8 heads) in one launch: F of KV head 0 and 5
    checked in full against the oracle, the LSE of every head at sampled rows."""
    w = kvp_inputs.QWEN3_4B_LAYER
    x = kvp_inputs.make_prefill(w, device="cuda")
    scale = w.head_dim ** -0.5
    lse, F = _run(kvp, x["q"], x["k"], w.window)
    q = x["q"][0].cpu()
    k = x["k"][0].cpu()
    G = w.group
    for h in (0, 5):
        qs, ks = q[h * G:(h + 1) * G], k[h:h + 1]
        lse_r = oracle.row_lse(qs, ks, scale)
        check_lse(np64(lse[0, h * G:(h + 1) * G]), lse_r, f"full h{h}")
        F_r = oracle.future_attn_mass(qs, ks, lse_r, scale, w.window)
        check_F(np64(F[0, h:h + 1]), F_r, f"full h{h}")
    rows = np.array([0, 1, 127, 128, 4095, 8064, 8190, 8191])
    lse_r = oracle.row_lse(q, k, scale, rows=rows)
    check_lse(np64(lse[0][:, rows]), lse_r, "full sampled rows")


def test_llama_32_layers_full_size(kvp):
    """Llama-3.1-8B-shaped: all 32 layers x 8 KV heads (S = 32768) in one launch; layers 0 and
    31 (KV head 0) checked in full, every F finite, non-negative, zero past S-1-w."""
    w = kvp_inputs.LLAMA31_8B_32L
    x = kvp_inputs.make_prefill(w, device="cuda")
    scale = w.head_dim ** -0.5
    lse, F = _run(kvp, x["q"], x["k"], w.window)
    S = w.seq_len
    assert torch.isfinite(F).all() and (F >= 0).all()
    assert (F[..., S - w.window:] == 0).all()
    G = w.group
    for layer in (0, 31):
        qs = x["q"][layer, :G].cpu()
        ks = x["k"][layer, :1].cpu()
        lse_r = oracle.row_lse(qs, ks, scale)
        check_lse(np64(lse[layer, :G]), lse_r, f"llama L{layer}")
        keys = np.unique(np.concatenate([np.arange(0, S, 97), np.arange(S - 2 * w.window, S)]))
        F_r = oracle.future_attn_mass(qs, ks, lse_r, scale, w.window, keys=keys)
        check_F(np64(F[layer, 0][keys])[None], F_r, f"llama L{layer}")


def test_qwen3_8b_131k_full_size(kvp):
    """S = 131072 in one launch: the late keys (whose future queries the oracle can afford)
    of KV head 3 in full, the LSE at sampled rows, and the properties that hold at any size."""
    w = kvp_inputs.QWEN3_8B_131K
    x = kvp_inputs.make_prefill(w, device="cuda")
    scale = w.head_dim ** -0.5
    lse, F = _run(kvp, x["q"], x["k"], w.window)
    S, G = w.seq_len, w.group
    assert torch.isfinite(F).all() and (F >= 0).all()
    assert (F[..., S - w.window:] == 0).all()
    j = torch.arange(S, device="cuda", dtype=torch.float32)
    assert (F[0] <= G * torch.clamp(S - j - w.window, min=0) * (1 + 1e-5)).all()
    h = 3
    qs = x["q"][0, h * G:(h + 1) * G].cpu()
    ks = x["k"][0, h:h + 1].cpu()
    first_q = S - 1536
    rows = np.arange(first_q, S)
    lse_rows = oracle.row_lse(qs, ks, scale, rows=rows)
    check_lse(np64(lse[0, h * G:(h + 1) * G])[:, rows], lse_rows, "131k late rows")
    sampled = np.array([0, 1, 2, 3, 4, 1000, 65535, 65536, 100000])
    check_lse(np64(lse[0, h * G:(h + 1) * G])[:, sampled],
              oracle.row_lse(qs, ks, scale, rows=sampled), "131k sampled rows")
    # keys whose every future query lies in `rows`: j >= first_q - w
    keys = np.arange(first_q - w.window, S)
    lse_full = np.zeros((G, S))
    lse_full[:, rows] = lse_rows
    F_r = oracle.future_attn_mass(qs, ks, lse_full, scale, w.window, keys=keys)
    check_F(np64(F[0, h])[keys][None], F_r, "131k late keys")


@pytest.mark.parametrize("step", [3.0, 50.0])
def test_growing_logits_lse(kvp, step):
    """Logits that grow along the key axis (natural-log slope `step` per 128 keys): the running
    normaliser must follow a maximum that keeps rising from tile to tile -- past 2^32 of its
    reference within a few tiles (step 3) and by more than 2^64 from one tile to the next
    (step 50, where F of the early keys is far below fp32's range and only the LSE is compared)."""
    S, Hq = 1100, 4
    gen = torch.Generator().manual_seed(int(step * 10))
    scale = 128 ** -0.5
    a = 8.0
    q = 0.05 * torch.randn(1, Hq, S, 128, generator=gen)
    q[..., 0] = a
    k = 0.05 * torch.randn(1, 1, S, 128, generator=gen)
    k[..., 0] = step * torch.arange(S, dtype=torch.float32) / (128 * scale * a)
    q, k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    lse, F = _run(kvp, q.cuda(), k.cuda(), 16)
    lse_r = oracle.row_lse(q[0], k[0], scale)
    assert lse_r[:, -1].min() > (300.0 if step > 10 else 20.0)
    check_lse(np64(lse[0]), lse_r, f"growing logits step {step}")
    if step < 10:
        F_r = oracle.future_attn_mass(q[0], k[0], lse_r, scale, 16)
        check_F(np64(F[0]), F_r, f"growing logits step {step}")


def _fused_qkv(B, S, Hq, Hkv, D, dtype, seed):
    """A fused QKV projection [B, S, (Hq + 2 Hkv) * D] and [B, H, S, D] views of its Q and K
    slices (head_dim contiguous, token stride (Hq + 2 Hkv) * D)."""
    gen = torch.Generator().manual_seed(seed)
    Ht = Hq + 2 * Hkv
    qkv = torch.randn(B, S, Ht, D, generator=gen).to(dtype)
    q = qkv[:, :, :Hq].permute(0, 2, 1, 3)
    k = qkv[:, :, Hq:Hq + Hkv].permute(0, 2, 1, 3)
    return qkv, q, k


@pytest.mark.parametrize("dtype,D,B", [(torch.bfloat16, 128, 1), (torch.float16, 64, 2),
                                       (torch.bfloat16, 64, 1), (torch.float32, 128, 2)])
def test_strided_fused_qkv_views(kvp, dtype, D, B):
    """Q and K read in place from a fused QKV buffer (token-major, heads interleaved) through the
    stride arguments: the same LSE and F as the oracle on dense copies, at a ragged S."""
    S, Hq, Hkv, w = 700, 8, 2, 32
    qkv, q, k = _fused_qkv(B, S, Hq, Hkv, D, dtype, seed=D + B)
    qkv_d = qkv.cuda()
    qv = qkv_d[:, :, :Hq].permute(0, 2, 1, 3)
    kv = qkv_d[:, :, Hq:Hq + Hkv].permute(0, 2, 1, 3)
    assert not qv.is_contiguous() and qv.stride(3) == 1 and qv.stride(2) == (Hq + 2 * Hkv) * D
    scale = D ** -0.5
    lse, F = _run(kvp, qv, kv, w)
    for b in range(B):
        lse_r, F_r = _oracle(q[b].contiguous(), k[b].contiguous(), w, scale)
        check_lse(np64(lse[b]), lse_r, f"strided {dtype} D{D} b{b}")
        check_F(np64(F[b]), F_r, f"strided {dtype} D{D} b{b}")
    # the dense copies give the same result (the stride path changes only the addressing)
    lse2, F2 = _run(kvp, qv.contiguous(), kv.contiguous(), w)
    assert torch.equal(lse, lse2) and torch.equal(F, F2)


def test_strided_sparse_lse_and_target(kvp):
    """The sparse row LSE and the KVpop target take the same stride arguments."""
    S, Hq, Hkv, D, w, n_sink, kk = 600, 4, 1, 128, 24, 4, 100
    qkv, q, k = _fused_qkv(1, S, Hq, Hkv, D, torch.bfloat16, seed=11)
    qkv_d = qkv.cuda()
    qv = qkv_d[:, :, :Hq].permute(0, 2, 1, 3)
    kv = qkv_d[:, :, Hq:Hq + Hkv].permute(0, 2, 1, 3)
    ranks = kvp_inputs.make_static_ranks(1, S, seed=3).reshape(1, Hkv, S)
    tau = kvp.kvp_topk_cutoffs(ranks.cuda(), n_sink, w, kk)
    lse_s = kvp.kvp_sparse_lse_pass(qv, kv, ranks.cuda(), tau, n_sink, w)
    lse_d = kvp.kvp_sparse_lse_pass(qv.contiguous(), kv.contiguous(), ranks.cuda(), tau, n_sink, w)
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    assert torch.equal(lse_s, lse_d)
    tgt_s, Fh_s, _ = kvp.kvp_future_attn_target(qv, kv, lse_s, w, want=("target", "F_heads"))
    tgt_d, Fh_d, _ = kvp.kvp_future_attn_target(qv.contiguous(), kv.contiguous(), lse_s, w,
                                                want=("target", "F_heads"))
    torch.cuda.synchronize()
    assert torch.equal(Fh_s, Fh_d) and torch.equal(tgt_s, tgt_d)
    scale = D ** -0.5
    tau_r = oracle.fenwick_cutoffs(ranks.numpy().reshape(S), n_sink, w, kk)[None]
    assert np.array_equal(tau.cpu().numpy().reshape(1, S), tau_r)
    q0, k0 = q[0].contiguous(), k[0].contiguous()
    lse_r = oracle.sparse_row_lse(q0, k0, ranks.numpy().reshape(Hkv, S), tau_r, scale, n_sink, w)
    check_lse(np64(lse_s[0]), lse_r, "strided sparse LSE")
    Fh_r = oracle.future_attn_mass_per_head(q0, k0, lse_r, scale, w)
    check_F(np64(Fh_s[0]), Fh_r, "strided target F_heads")


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.float16, 64), (torch.bfloat16, 64)])
def test_16bit_inputs_run_on_the_tensor_cores(kvp, dtype, D):
    """bf16 / f16 inputs run on the tcgen05 passes at head_dim 64 and 128 (there is no fp32
    fallback for them): on the Qwen3-4B-shaped layer the row-LSE pass runs faster than the
    fp32 FFMA pipes could score its pairs even at a 2.2 GHz clock (SMs x 128 FMA lanes x 2
    flops per clock), so the contraction ran on the tensor cores."""
    w = kvp_inputs.QWEN3_4B_LAYER.scaled(head_dim=D, dtype={torch.bfloat16: "bf16", torch.float16: "f16"}[dtype])
    x = kvp_inputs.make_prefill(w, device="cuda")
    lse = torch.empty(1, w.h_q, w.seq_len, device="cuda")
    for _ in range(3):
        kvp.kvp_lse_pass(x["q"], x["k"], lse=lse)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    times = []
    for _ in range(5):
        ev[0].record()
        kvp.kvp_lse_pass(x["q"], x["k"], lse=lse)
        ev[1].record()
        torch.cuda.synchronize()
        times.append(ev[0].elapsed_time(ev[1]) * 1e-3)
    kvp.kvp_check_device_status()
    S = w.seq_len
    flops = 2.0 * D * w.h_q * S * (S + 1) / 2
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ffma_peak = sms * 128 * 2 * 2.2e9
    assert flops / min(times) > 2.0 * ffma_peak, (flops / min(times) / 1e12, ffma_peak / 1e12)
    # and the result is the oracle's on a sampled head
    scale = D ** -0.5
    lse_r = oracle.row_lse(x["q"][0, :1].cpu(), x["k"][0, :1].cpu(), scale,
                           rows=np.array([0, 1, 500, 4096, S - 1]))
    check_lse(np64(lse[0, :1])[:, [0, 1, 500, 4096, S - 1]], lse_r, f"tc {dtype} D{D}")
