"""ctypes loader for libkvsel.so and the C ABI signatures of include/kvsel.h."""

from __future__ import annotations

import ctypes
import os
import threading

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkvsel.so")
_lock = threading.Lock()
_lib = None

c_i32, c_i64, c_u64, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p


class KvselShape(ctypes.Structure):
    """Mirror of ``kvsel_shape``."""
    _fields_ = [("num_layers", c_i32), ("num_seqs", c_i32), ("num_heads", c_i32),
                ("head_dim", c_i32), ("dtype", c_i32), ("num_kv_heads", c_i32),
                ("seq_offsets", ctypes.POINTER(c_i64))]


_P = ctypes.POINTER(KvselShape)

SIGNATURES = {
    "kvsel_version": (ctypes.c_char_p, []),
    "kvsel_status_string": (ctypes.c_char_p, [c_i32]),
    "kvsel_out_tokens": (c_i64, [_P, c_i32]),
    "kvsel_score_path": (c_i32, [_P, c_i32, c_i32]),
    "kvsel_window_logits": (c_i32, [_P, c_vp, c_vp, c_i32, c_vp, c_vp]),
    "kvsel_score": (c_i32, [_P, c_vp, c_vp, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp]),
    "kvsel_score_static": (c_i32, [_P, c_vp, c_vp, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp]),
    "kvsel_score_static_bytes": (c_i64, [_P, c_i32]),
    "kvsel_workspace_bytes": (c_i64, []),
    "kvsel_select": (c_i32, [_P, c_vp, c_i32, c_i32, c_vp, c_vp]),
    "kvsel_compact": (c_i32, [_P, c_vp, c_vp, c_vp, c_i32, c_vp, c_vp, c_vp]),
    "kvsel_snapkv": (c_i32, [_P, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp,
                             c_vp, c_vp]),
    "kvsel_snapkv_grouped": (c_i32, [_P, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_vp,
                                     c_vp, c_vp, c_vp]),
    "kvsel_snapkv_host": (c_i32, [_P, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp,
                                  c_vp, c_vp]),
    "kvsel_jacap_score": (c_i32, [_P, c_vp, c_vp, c_vp, c_i32, ctypes.c_float, ctypes.c_float,
                                  ctypes.c_float, c_vp, c_vp]),
    "kvsel_jacap": (c_i32, [_P, c_vp, c_vp, c_vp, c_i32, c_i32, ctypes.c_float, ctypes.c_float,
                            ctypes.c_float, c_vp, c_vp, c_vp, c_vp]),
    "kvsel_decode_attention": (c_i32, [_P, c_vp, c_vp, c_vp, c_i32, c_vp, c_vp, c_vp, c_vp,
                                       c_vp]),
    "kvsel_decode_quality": (c_i32, [c_i64, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "kvsel_reverse_attention": (c_i32, [_P, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "kvsel_cache_lengths": (c_i32, [_P, c_i32, c_i32, ctypes.POINTER(c_i64),
                                    ctypes.POINTER(c_i64)]),
    "kvsel_device_status": (c_i32, [c_vp]),
    "kvsel_set_wait_limit_ns": (c_i32, [c_u64]),
    "kvsel_debug_inject": (c_i32, [c_i32]),
    "kvsel_profile_begin": (c_i32, [c_i32]),
    "kvsel_profile_end": (c_i32, [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(c_i32)]),
    "kvsel_release": (None, []),
}


def lib_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built (there is no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is missing: build it with "
                    "`python -m kv_cache_eviction_snapkv_gb300.build`")
            handle = ctypes.CDLL(_LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
        return _lib
