"""The C-ABI library builds, loads and exports every symbol include/kvp.h declares;
host-side validation rejects bad arguments before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvp.h")


@pytest.fixture(scope="module")
def lib():
    from learned_kv_cache_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvp_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_five_stages():
    names = declared_functions()
    for n in ("kvp_lse_pass", "kvp_future_attn_mass", "kvp_select_topk", "kvp_compact_kv",
              "kvp_decode_attn"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_the_header():
    from learned_kv_cache_gb300 import _lib
    assert set(_lib.SIGNATURES) == set(declared_functions())


def test_missing_library_fails_loudly(tmp_path):
    from learned_kv_cache_gb300 import _lib
    saved = _lib._lib
    _lib._lib = None
    try:
        with pytest.raises(RuntimeError):
            _lib.load(str(tmp_path / "nope.so"))
    finally:
        _lib._lib = saved


def _bind(lib):
    from learned_kv_cache_gb300 import _lib
    for name, (res, args) in _lib.SIGNATURES.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    return lib


def test_host_validation_codes(lib):
    L = _bind(lib)
    p = ctypes.c_void_p(4096)     # never dereferenced: validation fails first
    assert L.kvp_abi_version() == 2
    assert L.kvp_status_string(-6) == b"device-side range check failed"
    # null pointer
    assert L.kvp_lse_pass(None, p, 1, 1, 4, 2, 16, 128, None, None, 0.1, p, None) == -1
    # unsupported head_dim / dtype
    assert L.kvp_lse_pass(p, p, 1, 1, 4, 2, 16, 96, None, None, 0.1, p, None) == -2
    assert L.kvp_lse_pass(p, p, 7, 1, 4, 2, 16, 128, None, None, 0.1, p, None) == -2
    assert b"dtype" in L.kvp_last_error()
    # GQA mismatch, misalignment, negative window
    assert L.kvp_lse_pass(p, p, 1, 1, 6, 4, 16, 128, None, None, 0.1, p, None) == -1
    assert L.kvp_lse_pass(ctypes.c_void_p(4098), p, 1, 1, 4, 2, 16, 128, None, None, 0.1, p, None) == -1
    assert L.kvp_future_attn_mass(p, p, p, 1, 1, 4, 2, 16, 128, None, None, 0.1, -1, p, None, 0, None) == -1
    # strides: not a multiple of 16 bytes, token stride below head_dim, non-positive
    for bad in ((4096, 128, 12), (4096, 128, 64), (0, 0, 0)):
        st = (ctypes.c_int64 * 3)(*bad)
        assert L.kvp_lse_pass(p, p, 1, 2, 4, 2, 16, 128, st, None, 0.1, p, None) == -1
        assert b"stride" in L.kvp_last_error()
    # select: stride < T, negative window sizes
    assert L.kvp_select_topk(p, 2, 100, 50, p, 4, 16, p, 64, p, None) == -1
    assert L.kvp_select_topk(p, 2, 100, 100, p, -1, 16, p, 64, p, None) == -1
    # soft-topk: k outside (0, n)
    assert L.kvp_soft_topk_budgets(p, 10, 10.0, 100, p, p, None) == -1
    assert L.kvp_soft_topk_budgets(p, 2000, 1.0, 100, p, p, None) == -1
    # decode: group too large, missing workspace
    assert L.kvp_decode_attn(p, p, p, 1, 1, 16, 1, 128, 64, p, 0.1, p, None, None, 0, 0, p, 1 << 30,
                             None) == -2
    assert L.kvp_decode_attn(p, p, p, 1, 1, 8, 2, 128, 64, p, 0.1, p, None, None, 0, 0, None, 0,
                             None) == -5
    # compact: bad head_dim
    assert L.kvp_compact_kv(p, p, 1, 2, 10, 32, p, p, 4, p, p, None) == -2


def test_workspace_queries(lib):
    L = _bind(lib)
    assert L.kvp_decode_attn_workspace_size(28, 12, 2, 128, 4096, 0) > 0
    with_mass = L.kvp_decode_attn_workspace_size(28, 12, 2, 128, 4096, 1)
    assert with_mass >= 56 * 6 * 4096 * 4
    assert L.kvp_decode_attn_workspace_size(28, 12, 5, 128, 4096, 0) == 0   # invalid -> 0
