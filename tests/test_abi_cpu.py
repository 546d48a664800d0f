"""C ABI checks that need no GPU: the library loads, exports every function
kvsel.h declares, and rejects bad arguments on the host before any launch."""

import ctypes
import os
import re
import subprocess

import pytest

from helpers import ROOT, ensure_built


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    from kv_cache_eviction_snapkv_gb300 import _native
    return _native.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "kvsel.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvsel_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["kvsel_score", "kvsel_select", "kvsel_compact", "kvsel_snapkv",
              "kvsel_device_status", "kvsel_status_string", "kvsel_out_tokens"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from kv_cache_eviction_snapkv_gb300 import _native
    out = subprocess.run(["nm", "-D", "--defined-only", _native.lib_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (kvsel_\w+)", out))
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(lib, n)
        assert n in _native.SIGNATURES, f"binding lacks {n}"


def test_library_has_sm103a_code_and_no_host_driver_dependency(lib):
    from kv_cache_eviction_snapkv_gb300 import _native
    out = subprocess.run(["readelf", "-d", _native.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    assert "libcuda.so" not in out          # driver resolved at run time only
    assert "libcudart.so" not in out        # runtime linked statically


def test_status_strings_and_version(lib):
    from kv_cache_eviction_snapkv_gb300 import api
    assert "sm_103a" in api.kvsel_version()
    assert api.kvsel_status_string(0) == "ok"
    assert "index" in api.kvsel_status_string(api.KVSEL_ERR_BAD_INDEX)
    assert api.kvsel_status_string(99) == "unknown status"


def test_out_tokens(lib):
    from kv_cache_eviction_snapkv_gb300 import api
    sh = api.Shape(2, 4, 128, api.KVSEL_BF16, [0, 100, 130, 5130])
    assert api.kvsel_out_tokens(sh, 64) == 64 + 30 + 64
    assert api.kvsel_out_tokens(sh, 1000) == 100 + 30 + 1000
    assert api.kvsel_out_tokens(sh, 0) == -1
    assert api.kvsel_out_tokens(api.Shape(1, 1, 1, 0, [0]), 5) == 0
    assert api.kvsel_out_tokens(api.Shape(1, 1, 1, 0, [0, 5, 3]), 5) == -1   # decreasing
    assert api.kvsel_out_tokens(api.Shape(1, 1, 1, 0, [1, 5]), 5) == -1      # offsets[0] != 0
    assert api.kvsel_out_tokens(api.Shape(1, 1, 1, 7, [0, 5]), 5) == -1      # dtype


def _call_snapkv(lib, shape, W, C, kind=0, k=3, ptrs=True):
    p = ctypes.c_void_p(0x1000) if ptrs else None
    return lib.kvsel_snapkv(ctypes.byref(shape.c), p, p, p, W, C, kind, k, p, p, p, None)


@pytest.mark.parametrize("case,expect", [
    (dict(W=0), 1), (dict(C=32), 1), (dict(C=10), 1), (dict(W=200), 1),
    (dict(kind=2), 1), (dict(k=4), 1), (dict(k=0), 1), (dict(C=20000), 2),
    (dict(ptrs=False), 1),
])
def test_snapkv_argument_rules(lib, case, expect):
    """Rejected on the host (no GPU touched): W >= 1, C > W, W <= L_b for every
    sequence, pooling kind, odd positive width, non-null pointers, C - W limit."""
    from kv_cache_eviction_snapkv_gb300 import api
    sh = api.Shape(1, 2, 64, api.KVSEL_BF16, [0, 100, 300])
    W = case.get("W", 32)
    C = case.get("C", 64)
    if case.get("W") == 200:
        C = 300
    assert _call_snapkv(lib, sh, W, C, case.get("kind", 0), case.get("k", 3),
                        case.get("ptrs", True)) == expect


def test_other_entry_points_reject_on_host(lib):
    from kv_cache_eviction_snapkv_gb300 import api
    sh = api.Shape(1, 2, 64, api.KVSEL_BF16, [0, 100, 300])
    p = ctypes.c_void_p(0x1000)
    assert lib.kvsel_score(ctypes.byref(sh.c), p, p, 0, 0, 3, p, p, None) == 1
    assert lib.kvsel_score(ctypes.byref(sh.c), p, p, 8, 0, 2, p, p, None) == 1
    assert lib.kvsel_score(ctypes.byref(sh.c), p, p, 8, 0, 3, p, None, None) == 1
    assert lib.kvsel_select(ctypes.byref(sh.c), p, 8, 8, p, None) == 1
    assert lib.kvsel_compact(ctypes.byref(sh.c), p, p, p, 0, p, p, None) == 1
    assert lib.kvsel_compact(ctypes.byref(sh.c), None, p, p, 64, p, p, None) == 1
    assert lib.kvsel_window_logits(ctypes.byref(sh.c), p, p, 101, p, None) == 1
    bad = api.Shape(1, 2, 64, api.KVSEL_BF16, [0, 100, 300])
    bad.c.num_kv_heads = 3                       # must divide num_heads
    assert lib.kvsel_window_logits(ctypes.byref(bad.c), p, p, 8, p, None) == 1
    bad.c.num_kv_heads = -1
    assert lib.kvsel_snapkv(ctypes.byref(bad.c), p, p, p, 8, 16, 0, 3, p, p, p, None) == 1
    assert lib.kvsel_snapkv_grouped(ctypes.byref(bad.c), p, p, p, 8, 16, 0, 3, p, p, p,
                                    None) == 1
    gqa = api.Shape(1, 4, 64, api.KVSEL_BF16, [0, 100, 300], num_kv_heads=2)
    assert gqa.c.num_kv_heads == 2
    assert lib.kvsel_snapkv_grouped(ctypes.byref(gqa.c), p, p, p, 8, 8, 0, 3, p, p, p,
                                    None) == 1      # C must exceed W
    assert lib.kvsel_set_wait_limit_ns(10) == 1
    assert lib.kvsel_debug_inject(5) == 1


def test_empty_batch_is_a_noop(lib):
    from kv_cache_eviction_snapkv_gb300 import api
    sh = api.Shape(3, 4, 128, api.KVSEL_BF16, [0])
    assert _call_snapkv(lib, sh, 8, 16, ptrs=False) == 0


def test_decode_entry_points_host_rules(lib):
    """Argument rules of the decode entry points (checked before any device work)."""
    from kv_cache_eviction_snapkv_gb300 import api
    p = ctypes.c_void_p(256)
    sh = api.Shape(1, 4, 128, api.KVSEL_BF16, [0, 100, 130])
    assert lib.kvsel_decode_attention(ctypes.byref(sh.c), p, p, p, -1, p, p, p, p, None) == 1
    assert lib.kvsel_decode_attention(ctypes.byref(sh.c), None, p, p, 0, None, None, p, p,
                                      None) == 1
    assert lib.kvsel_decode_attention(ctypes.byref(sh.c), p, p, p, 3, None, None, p, p,
                                      None) == 1            # g > 0 needs K_new, V_new
    odd = ctypes.c_void_p(258)
    assert lib.kvsel_decode_attention(ctypes.byref(sh.c), odd, p, p, 0, None, None, p, p,
                                      None) == 1            # 16-byte alignment
    d96 = api.Shape(1, 4, 96, api.KVSEL_BF16, [0, 100])
    assert lib.kvsel_decode_attention(ctypes.byref(d96.c), p, p, p, 0, None, None, p, p,
                                      None) == 2            # D not in {64, 128}
    empty_seq = api.Shape(1, 4, 128, api.KVSEL_BF16, [0, 100, 100])
    assert lib.kvsel_decode_attention(ctypes.byref(empty_seq.c), p, p, p, 0, None, None, p, p,
                                      None) == 1            # a sequence with no rows at all
    assert lib.kvsel_decode_quality(-1, 128, p, p, p, p, p, p, None) == 1
    assert lib.kvsel_decode_quality(5, 0, p, p, p, p, p, p, None) == 1
    assert lib.kvsel_decode_quality(5, 128, None, p, p, p, p, p, None) == 1
    assert lib.kvsel_decode_quality(0, 128, None, None, None, None, None, None, None) == 0


def test_cache_lengths_follow_the_page(lib):
    """min(L, C) + g physical rows and L + g logical positions (host only)."""
    from kv_cache_eviction_snapkv_gb300 import api
    phys, logi = api.kvsel_cache_lengths([0, 8, 11, 5011], 5, 0)
    assert phys == [5, 3, 5] and logi == [8, 3, 5000]
    phys, logi = api.kvsel_cache_lengths([0, 8, 11, 5011], 5, 7)
    assert phys == [12, 10, 12] and logi == [15, 10, 5007]
    sh = api.Shape(1, 1, 1, api.KVSEL_BF16, [0, 8])
    assert lib.kvsel_cache_lengths(ctypes.byref(sh.c), 0, 0, None, None) == 1
    assert lib.kvsel_cache_lengths(ctypes.byref(sh.c), 5, -1, None, None) == 1


def test_jacap_host_rules(lib):
    """Jacap argument rules and the tensor-path limits, checked on the host."""
    from kv_cache_eviction_snapkv_gb300 import api
    p = ctypes.c_void_p(256)
    f = ctypes.c_float
    sh = api.Shape(1, 4, 128, api.KVSEL_BF16, [0, 1000, 1500])
    assert lib.kvsel_jacap_score(ctypes.byref(sh.c), p, p, p, 0, f(10), f(0.9), f(1e-6), p,
                                 None) == 1                      # W = 0
    assert lib.kvsel_jacap_score(ctypes.byref(sh.c), p, p, p, 8, f(0), f(0.9), f(1e-6), p,
                                 None) == 1                      # tau
    assert lib.kvsel_jacap_score(ctypes.byref(sh.c), p, p, p, 8, f(10), f(1.0), f(1e-6), p,
                                 None) == 1                      # beta
    assert lib.kvsel_jacap_score(ctypes.byref(sh.c), p, p, p, 8, f(10), f(0.5), f(-1), p,
                                 None) == 1                      # eps
    d64 = api.Shape(1, 4, 64, api.KVSEL_BF16, [0, 1000])
    assert lib.kvsel_jacap_score(ctypes.byref(d64.c), p, p, p, 8, f(10), f(0.9), f(1e-6), p,
                                 None) == 2                      # D = 64: no tensor path
    gqa = api.Shape(1, 4, 128, api.KVSEL_BF16, [0, 1000], num_kv_heads=2)
    assert lib.kvsel_jacap_score(ctypes.byref(gqa.c), p, p, p, 8, f(10), f(0.9), f(1e-6), p,
                                 None) == 2                      # grouped K/V heads
    assert lib.kvsel_jacap(ctypes.byref(sh.c), p, p, p, 8, 8, f(10), f(0.9), f(1e-6), p, p, p,
                           None) == 1                            # C <= W


def test_reverse_host_rules(lib):
    """Reverse-mask attention: argument rules and the tensor-path limits, on the host."""
    from kv_cache_eviction_snapkv_gb300 import api
    p = ctypes.c_void_p(256)
    sh = api.Shape(1, 4, 128, api.KVSEL_BF16, [0, 300, 301], num_kv_heads=2)
    assert lib.kvsel_reverse_attention(ctypes.byref(sh.c), None, p, p, None, p, None,
                                       None) == 1                  # Q missing
    assert lib.kvsel_reverse_attention(ctypes.byref(sh.c), p, p, p, None, None, None,
                                       None) == 1                  # out missing
    assert lib.kvsel_reverse_attention(ctypes.byref(sh.c), p, p, p, None, ctypes.c_void_p(260),
                                       None, None) == 1            # out misaligned
    d64 = api.Shape(1, 4, 64, api.KVSEL_BF16, [0, 300])
    assert lib.kvsel_reverse_attention(ctypes.byref(d64.c), p, p, p, None, p, None,
                                       None) == 2                  # D = 64
    f32 = api.Shape(1, 4, 128, api.KVSEL_F32, [0, 300])
    assert lib.kvsel_reverse_attention(ctypes.byref(f32.c), p, p, p, None, p, None,
                                       None) == 2                  # fp32
    bad = api.Shape(1, 4, 128, api.KVSEL_BF16, [0, 300, 200])
    assert lib.kvsel_reverse_attention(ctypes.byref(bad.c), p, p, p, None, p, None,
                                       None) == 1                  # decreasing offsets
    empty = api.Shape(1, 4, 128, api.KVSEL_BF16, [0, 0])
    assert lib.kvsel_reverse_attention(ctypes.byref(empty.c), None, None, None, None, None, None,
                                       None) == 0                  # nothing to do


def test_binding_arity_matches_the_header():
    """Every declaration's parameter count equals its ctypes signature's."""
    from kv_cache_eviction_snapkv_gb300 import _native
    text = open(os.path.join(ROOT, "include", "kvsel.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    decls = re.findall(r"\b(kvsel_[a-z_]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S)
    assert decls
    for name, params in decls:
        params = " ".join(params.split())
        n = 0 if params in ("", "void") else params.count(",") + 1
        assert len(_native.SIGNATURES[name][1]) == n, (name, n)
