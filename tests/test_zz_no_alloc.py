"""kvp_decode_attn_noalloc: the decode entry point for callers that cannot allocate device
memory (a host whose HBM is already reserved by its own pool, a plain-C program with no
device allocator, a decode loop that must not call cudaMalloc/cudaFree because they can
synchronise the device).  It uses the library's fixed per-device scratch instead of a
caller workspace.

Called here directly through the C ABI (ctypes), on two calls in a row per shape (the
second call finds the first call's partials still in the shared scratch), and checked
* against the fp64 oracle (max abs 2e-3), which shares nothing with the CUDA path;
* against kvp_decode_attn, which takes a caller workspace;
* for allocating nothing: after a warm-up call, the device's free memory is the same before
  and after a call.
Three shapes: the Qwen2.5-1.5B-shaped pruned cache (fp16, tensor-core decode), a bf16 cache
with ragged lengths, and a float32 cache (the fp32 split-K decode, whose partials also live
in the scratch).

This file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import DECODE_ATOL

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, q, kc, vc, lens, out):
    L, Hq, D = q.shape
    R, T_cap, _ = kc.shape
    dt = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}[q.dtype]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.kvp_decode_attn_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kc.data_ptr()), ctypes.c_void_p(vc.data_ptr()),
        dt, L, Hq, R // L, D, T_cap, ctypes.c_void_p(lens.data_ptr()), D ** -0.5,
        ctypes.c_void_p(out.data_ptr()), stream)


CASES = [
    # Qwen2.5-1.5B-shaped pruned cache (28 layers, 12/2 heads, fp16, 4096 kept per row)
    (28, 12, 2, 128, 4096, torch.float16, 0),
    # a different shape and dtype with ragged lengths, reusing the same scratch
    (3, 8, 2, 64, 1500, torch.bfloat16, 1),
    # float32 cache: the fp32 split-K decode
    (2, 6, 3, 128, 2500, torch.float32, 2),
]


def test_noalloc_decode_matches_oracle_and_workspace_decode_twice():
    import learned_kv_cache_gb300 as kvp
    lib = kvp.load()
    dev = "cuda"
    for L, Hq, Hkv, D, T_cap, dt, seed in CASES:
        gen = torch.Generator(device=dev).manual_seed(seed)
        R = L * Hkv
        q = torch.randn(L, Hq, D, generator=gen, device=dev).to(dt)
        kc = torch.randn(R, T_cap, D, generator=gen, device=dev).to(dt)
        vc = torch.randn(R, T_cap, D, generator=gen, device=dev).to(dt)
        lens = torch.randint(0, T_cap + 1, (R,), generator=gen, device=dev, dtype=torch.int32)
        lens[0] = T_cap
        want, _ = oracle.decode_attn(q.cpu(), kc.cpu(), vc.cpu(), lens.cpu().numpy(), D ** -0.5)
        ws_out = kvp.kvp_decode_attn(q, kc, vc, lens)
        outs = [torch.full((L, Hq, D), float("nan"), device=dev) for _ in range(2)]
        torch.cuda.synchronize()
        for call, out in enumerate(outs):
            free0 = torch.cuda.mem_get_info()[0]
            rc = _call_noalloc(lib, q, kc, vc, lens, out)
            assert rc == 0, lib.kvp_last_error()
            torch.cuda.synchronize()
            free1 = torch.cuda.mem_get_info()[0]
            kvp.kvp_check_device_status()
            if call == 1:   # the first call may load the module (and place the fixed array)
                assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
            got = out.double().cpu().numpy()
            assert np.isfinite(got).all()
            err = np.abs(got - want).max()
            assert err <= DECODE_ATOL, (dt, call, err)
            err_ws = (out.double() - ws_out.double()).abs().max().item()
            assert err_ws <= DECODE_ATOL, (dt, call, err_ws)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import learned_kv_cache_gb300 as kvp
    lib = kvp.load()
    # 28 layers x 2 KV heads x 6 query heads over a 2,000,000-token cache needs far more
    # partials than the built-in scratch holds: rejected before any launch.
    L, Hq, Hkv, D, T_cap = 28, 12, 2, 128, 2_000_000
    dummy = torch.zeros(16, device="cuda", dtype=torch.float16)
    lens = torch.zeros(L * Hkv, device="cuda", dtype=torch.int32)
    out = torch.zeros(1, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.kvp_decode_attn_noalloc(ctypes.c_void_p(dummy.data_ptr()), ctypes.c_void_p(dummy.data_ptr()),
                                     ctypes.c_void_p(dummy.data_ptr()), 2, L, Hq, Hkv, D, T_cap,
                                     ctypes.c_void_p(lens.data_ptr()), D ** -0.5,
                                     ctypes.c_void_p(out.data_ptr()), stream)
    assert rc == -5
    assert b"scratch" in lib.kvp_last_error()
