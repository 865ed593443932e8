"""GPU parity of chunked prefill-compress (kvp_chunk_compress) against the oracle, step by
step and bit-exact: kept indices, counts, K/V bytes, scores and source positions; and the final
cache against one selection over the whole prefix."""
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


def _run_loop(kvp, k, v, s, C, b, ns, nr):
    R, S, D = k.shape
    dev = "cuda"
    cap = max(b, ns + nr)
    bufs = [{"k": torch.empty(R, cap, D, dtype=k.dtype, device=dev),
             "v": torch.empty(R, cap, D, dtype=k.dtype, device=dev),
             "score": torch.empty(R, cap, device=dev),
             "pos": torch.empty(R, cap, dtype=torch.int32, device=dev)} for _ in range(2)]
    kd, vd, sd = k.to(dev), v.to(dev), s.to(dev)
    cache, n, ref, ref_n = None, 0, None, 0
    for step, p0 in enumerate(range(0, S, C)):
        p1 = min(S, p0 + C)
        out = bufs[step % 2]
        idx, cnt = kvp.kvp_chunk_compress(cache, n, kd[:, p0:p1].contiguous(), vd[:, p0:p1].contiguous(),
                                          sd[:, p0:p1].contiguous(), p0, b, ns, nr, out)
        torch.cuda.synchronize()
        kvp.kvp_check_device_status()
        ref, ridx, rcnt = oracle.chunk_compress_step(
            ref, ref_n, k[:, p0:p1].view(torch.int16).numpy(), v[:, p0:p1].view(torch.int16).numpy(),
            s[:, p0:p1].numpy(), p0, b, ns, nr)
        got_cnt = cnt.cpu().numpy()
        assert (got_cnt == rcnt).all(), f"step {step}"
        m = int(rcnt[0])
        assert (idx.cpu().numpy()[:, :m] == ridx[:, :m]).all(), f"step {step}"
        assert (out["k"][:, :m].cpu().view(torch.int16).numpy() == ref["k"]).all()
        assert (out["v"][:, :m].cpu().view(torch.int16).numpy() == ref["v"]).all()
        assert (out["score"][:, :m].cpu().numpy() == ref["score"]).all()
        assert (out["pos"][:, :m].cpu().numpy() == ref["pos"]).all()
        cache, n, ref_n = out, m, m
    return cache, n


@pytest.mark.parametrize("dtype,D,S,C,b,ns,nr,ties", [
    ("bf16", 128, 5000, 1024, 1024, 4, 64, False),
    ("f16", 128, 3000, 16, 300, 4, 64, False),      # chunks shorter than the recent window
    ("bf16", 64, 2100, 700, 256, 2, 32, True),      # heavy score ties
    ("f16", 128, 900, 2000, 4096, 4, 64, False),    # one chunk, everything kept
])
def test_chunked_prefill_compress_matches_oracle(kvp, dtype, D, S, C, b, ns, nr, ties):
    R = 6
    gen = torch.Generator().manual_seed(S + C)
    dt = kvp_inputs.torch_dtype(dtype)
    k = torch.randn(R, S, D, generator=gen).to(dt)
    v = torch.randn(R, S, D, generator=gen).to(dt)
    s = kvp_inputs.make_scores(R, S, seed=S + b, quantize=2 if ties else None)
    cache, n = _run_loop(kvp, k, v, s, C, b, ns, nr)
    for r in range(R):
        keep = oracle.select_row(s[r].numpy().astype(np.float64), b, ns, nr)
        assert n == keep.size
        assert (cache["pos"][r, :n].cpu().numpy() == keep).all()


def test_chunk_compress_rejects_small_output(kvp):
    R, C, D = 2, 64, 128
    ck = torch.zeros(R, C, D, dtype=torch.bfloat16, device="cuda")
    cs = torch.zeros(R, C, device="cuda")
    out = {"k": torch.empty(R, 8, D, dtype=torch.bfloat16, device="cuda"),
           "v": torch.empty(R, 8, D, dtype=torch.bfloat16, device="cuda"),
           "score": torch.empty(R, 8, device="cuda"), "pos": torch.empty(R, 8, dtype=torch.int32, device="cuda")}
    with pytest.raises(kvp.KvpError):
        kvp.kvp_chunk_compress(None, 0, ck, ck, cs, 0, 32, 4, 8, out)


def test_chunked_budget_below_sinks_plus_window(kvp):
    """budget < n_sink + n_recent: every step keeps n_sink + n_recent entries (the effective budget)."""
    R, D, S, C, b, ns, nr = 3, 64, 700, 100, 10, 4, 32
    gen = torch.Generator().manual_seed(5)
    k = torch.randn(R, S, D, generator=gen).to(torch.float16)
    v = torch.randn(R, S, D, generator=gen).to(torch.float16)
    s = kvp_inputs.make_scores(R, S, seed=11)
    cache, n = _run_loop(kvp, k, v, s, C, b, ns, nr)
    assert n == ns + nr
