"""GPU parity of the static (ring) cache: a stream of decode steps, each inserting the new
token in place (kvp_ring_insert) and then attending over the cache while accumulating every
slot's attention (kvp_decode_attn key mass), checked step by step against the oracle.

The slot choice is an integer decided by fp32 scores, so the oracle decides on the GPU's
scores (the same precision); slots, positions and cache bytes must then agree exactly, the
decode output within 2e-3 and the accumulated scores within 2e-3 relative (+1e-6)."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import DECODE_ATOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvp():
    import learned_kv_cache_gb300 as m
    m.load()
    return m


@pytest.mark.parametrize("dtype,D,cap,n_sink,n_recent,steps", [
    (torch.float16, 128, 48, 4, 8, 160),
    (torch.bfloat16, 64, 32, 2, 3, 120),
    (torch.bfloat16, 128, 37, 1, 5, 100),
])
def test_ring_stream_matches_oracle(kvp, dtype, D, cap, n_sink, n_recent, steps):
    L, Hkv, G = 2, 2, 3
    R, Hq = L * Hkv, Hkv * G
    dev = "cuda"
    gen = torch.Generator().manual_seed(D + cap)
    toks_k = torch.randn(steps, R, D, generator=gen).to(dtype)
    toks_v = torch.randn(steps, R, D, generator=gen).to(dtype)
    qs = (torch.randn(steps, L, Hq, D, generator=gen) * 2).to(dtype)
    kc = torch.zeros(R, cap, D, dtype=dtype, device=dev)
    vc = torch.zeros_like(kc)
    pos = torch.full((R, cap), -1, dtype=torch.int32, device=dev)
    score = torch.zeros(R, cap, device=dev)
    fill = torch.zeros(R, dtype=torch.int32, device=dev)
    slot = torch.empty(R, dtype=torch.int32, device=dev)
    view = torch.int16
    r_kc = np.zeros((R, cap, D), dtype=np.int16)
    r_vc = np.zeros((R, cap, D), dtype=np.int16)
    r_pos = np.full((R, cap), -1)
    r_fill = np.zeros(R, dtype=np.int64)
    scale = D ** -0.5
    for t in range(steps):
        gpu_scores = score.cpu().numpy().astype(np.float64)          # scores the step decides on
        nk, nv = toks_k[t].to(dev), toks_v[t].to(dev)
        kvp.kvp_ring_insert(kc, vc, pos, score, fill, nk, nv, t, n_sink, n_recent, out_slot=slot)
        out = kvp.kvp_decode_attn(qs[t].to(dev), kc, vc, fill, key_mass=score, accumulate=True)
        torch.cuda.synchronize()
        kvp.kvp_check_device_status()
        r_score = gpu_scores.copy()
        want_slots = oracle.ring_insert(r_kc, r_vc, r_pos, r_score, r_fill,
                                        toks_k[t].view(view).numpy(), toks_v[t].view(view).numpy(),
                                        t, n_sink, n_recent)
        assert slot.cpu().numpy().tolist() == want_slots.tolist(), f"step {t}"
        assert (pos.cpu().numpy() == r_pos).all()
        assert (fill.cpu().numpy() == r_fill).all()
        assert kc.cpu().view(view).numpy().tobytes() == r_kc.tobytes()
        assert vc.cpu().view(view).numpy().tobytes() == r_vc.tobytes()
        kf = torch.from_numpy(r_kc).view(dtype)
        vf = torch.from_numpy(r_vc).view(dtype)
        ref, mass = oracle.decode_attn(qs[t], kf, vf, r_fill, scale)
        assert np.abs(out.cpu().double().numpy() - ref).max() <= DECODE_ATOL, f"step {t}"
        want_score = r_score + mass
        got_score = score.cpu().numpy()
        live = np.arange(cap)[None, :] < r_fill[:, None]
        assert (np.abs(got_score - want_score)[live] <= 2e-3 * np.abs(want_score[live]) + 1e-6).all()


def test_ring_rejects_small_capacity(kvp):
    kc = torch.zeros(1, 4, 128, dtype=torch.float16, device="cuda")
    pos = torch.zeros(1, 4, dtype=torch.int32, device="cuda")
    sc = torch.zeros(1, 4, device="cuda")
    fill = torch.zeros(1, dtype=torch.int32, device="cuda")
    nk = torch.zeros(1, 128, dtype=torch.float16, device="cuda")
    with pytest.raises(kvp.KvpError):
        kvp.kvp_ring_insert(kc, kc, pos, sc, fill, nk, nk, 0, 2, 3)
