"""GPU parity of the KVpop target (per-query-head future mass, count normalisation, log and
group aggregation) against the fp64 oracle.

Tolerances: per-head mass as F (2e-3 relative, exact zeros); the target is a log of the
count-normalised mass, so a relative error e of the mass is an absolute error ~e of the
target: 2e-3 absolute on finite entries, identical -inf where a key receives no mass."""
import numpy as np
import pytest
import torch

import kvp_inputs
import oracle
from tests.gpu_util import F_RTOL, check_F, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvp():
    import learned_kv_cache_gb300 as m
    m.load()
    return m


def check_target(got, want, what):
    got = np.asarray(got, np.float64)
    inf = np.isneginf(want)
    assert (np.isneginf(got) == inf).all(), f"{what}: -inf pattern differs"
    err = np.abs(got[~inf] - want[~inf]).max() if (~inf).any() else 0.0
    assert err <= F_RTOL, f"{what}: target max abs err {err:.3e}"


def _run(kvp, q, k, w, eps, agg):
    lse = kvp.kvp_lse_pass(q, k)
    tgt, Fh, F = kvp.kvp_future_attn_target(q, k, lse, w, eps=eps, aggregate=agg,
                                            want=("target", "F_heads", "F"))
    torch.cuda.synchronize()
    kvp.kvp_check_device_status()
    return tgt, Fh, F


def _oracle(q, k, w, G, eps, agg):
    scale = q.shape[-1] ** -0.5
    lse = oracle.row_lse(q, k, scale)
    Fh = oracle.future_attn_mass_per_head(q, k, lse, scale, w)
    return oracle.kvpop_target(Fh, w, G, eps=eps, aggregate=agg), Fh


@pytest.mark.parametrize("agg", ["max_log", "mean_prob"])
@pytest.mark.parametrize("dtype,D", [("f32", 64), ("bf16", 128), ("f16", 128), ("bf16", 64)])
def test_target_reduced_qwen3_recipe(kvp, dtype, D, agg):
    w = kvp_inputs.QWEN3_4B_LAYER.scaled(seq_len=700, head_dim=D, dtype=dtype, h_q=8, h_kv=2)
    x = kvp_inputs.make_prefill(w)
    tgt, Fh, F = _run(kvp, x["q"].cuda(), x["k"].cuda(), w.window, 0.0, agg)
    t_ref, Fh_ref = _oracle(x["q"][0], x["k"][0], w.window, w.group, 0.0, agg)
    check_F(np64(Fh[0]), Fh_ref, f"{dtype} D{D} per-head")
    check_F(np64(F[0]), Fh_ref.reshape(w.h_kv, w.group, -1).sum(1), f"{dtype} D{D} sum")
    check_target(np64(tgt[0]), t_ref, f"{dtype} D{D} {agg}")


def test_target_tiny_workload_with_eps(kvp):
    w = kvp_inputs.TINY
    x = kvp_inputs.make_prefill(w)
    tgt, Fh, F = _run(kvp, x["q"].cuda(), x["k"].cuda(), w.window, 1e-6, "max_log")
    t_ref, Fh_ref = _oracle(x["q"][0], x["k"][0], w.window, w.group, 1e-6, "max_log")
    check_F(np64(Fh[0]), Fh_ref, "tiny per-head")
    check_target(np64(tgt[0]), t_ref, "tiny")


@pytest.mark.parametrize("S,w", [(1, 0), (50, 60), (130, 129), (257, 0)])
def test_target_edges(kvp, S, w):
    gen = torch.Generator().manual_seed(S + w)
    q = torch.randn(1, 4, S, 128, generator=gen).to(torch.bfloat16)
    k = torch.randn(1, 2, S, 128, generator=gen).to(torch.bfloat16)
    tgt, Fh, F = _run(kvp, q.cuda(), k.cuda(), w, 0.0, "max_log")
    t_ref, Fh_ref = _oracle(q[0], k[0], w, 2, 0.0, "max_log")
    check_F(np64(Fh[0]), Fh_ref, f"edge S{S} w{w}")
    check_target(np64(tgt[0]), t_ref, f"edge S{S} w{w}")


def test_target_qwen3_4b_layer_full_size(kvp):
    """S = 8192, 32/8 heads in one launch; KV head 2 (4 query heads) in full."""
    w = kvp_inputs.QWEN3_4B_LAYER
    x = kvp_inputs.make_prefill(w, device="cuda")
    tgt, Fh, F = _run(kvp, x["q"], x["k"], w.window, 0.0, "max_log")
    G, h = w.group, 2
    qs = x["q"][0, h * G:(h + 1) * G].cpu()
    ks = x["k"][0, h:h + 1].cpu()
    t_ref, Fh_ref = _oracle(qs, ks, w.window, G, 0.0, "max_log")
    check_F(np64(Fh[0, h * G:(h + 1) * G]), Fh_ref, "full per-head")
    check_target(np64(tgt[0, h:h + 1]), t_ref, "full target")
