"""Thin Python binding of libkvsel: the C ABI's names, torch tensors in and out.

Argument marshalling only: every step of the selection runs in the library's
CUDA kernels. Tensors must be CUDA, contiguous, and laid out as ``kvsel.h``
states:

    q_win  [layers, S*W, H, D]      K, V  [layers, T, H, D]      (bf16 or fp32)
    votes, pooled [layers, H, T] fp32
    out_idx [layers, T_out, H] int32     out_K, out_V [layers, T_out, H, D]

3-D tensors (no layer axis) are accepted as one layer. ``seq_offsets`` is a
host sequence of S + 1 token offsets. Work is queued on the current torch
stream (or ``stream``); call ``kvsel_device_status`` to learn about errors
only the GPU can see.
"""

from __future__ import annotations

import ctypes
from typing import Optional, Sequence, Tuple

import torch

from . import _native

KVSEL_OK = 0
KVSEL_ERR_INVALID_ARG = 1
KVSEL_ERR_UNSUPPORTED = 2
KVSEL_ERR_NONFINITE = 3
KVSEL_ERR_TIMEOUT = 4
KVSEL_ERR_CUDA = 5
KVSEL_ERR_BAD_INDEX = 6
KVSEL_POOL_AVG = 0
KVSEL_POOL_MAX = 1
KVSEL_BF16 = 0
KVSEL_F32 = 1

_DTYPES = {torch.bfloat16: KVSEL_BF16, torch.float32: KVSEL_F32}


class KvselError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {kvsel_status_string(status)} (status {status})")


def _check(status: int, where: str) -> None:
    if status != KVSEL_OK:
        raise KvselError(status, where)


def kvsel_version() -> str:
    return _native.lib().kvsel_version().decode()


def kvsel_status_string(status: int) -> str:
    return _native.lib().kvsel_status_string(int(status)).decode()


class Shape:
    """Builds a ``kvsel_shape`` and keeps its host offsets alive."""

    def __init__(self, num_layers: int, num_heads: int, head_dim: int, dtype: int,
                 seq_offsets: Sequence[int], num_kv_heads: int = 0):
        offs = [int(x) for x in seq_offsets]
        self._offs = (ctypes.c_int64 * max(1, len(offs)))(*offs)
        kv = 0 if int(num_kv_heads) == int(num_heads) else int(num_kv_heads)
        self.c = _native.KvselShape(int(num_layers), len(offs) - 1, int(num_heads),
                                    int(head_dim), int(dtype), kv,
                                    ctypes.cast(self._offs, ctypes.POINTER(ctypes.c_int64)))
        self.T = offs[-1] if offs else 0

    @property
    def ref(self):
        return ctypes.byref(self.c)


def _as4(t: torch.Tensor) -> torch.Tensor:
    return t.unsqueeze(0) if t.dim() == 3 else t


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _need(t: torch.Tensor, name: str, dtype=None) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")


def shape_of(K: torch.Tensor, seq_offsets: Sequence[int], num_heads: Optional[int] = None
             ) -> Shape:
    """Shape of a call on K [layers, T, H_kv, D]; num_heads = the query (and
    per-head output) heads, default H_kv (no grouped-query attention)."""
    K4 = _as4(K)
    if K4.dtype not in _DTYPES:
        raise ValueError("K must be bf16 or fp32")
    h = K4.shape[2] if num_heads is None else int(num_heads)
    return Shape(K4.shape[0], h, K4.shape[3], _DTYPES[K4.dtype], seq_offsets,
                 num_kv_heads=K4.shape[2])


def kvsel_out_tokens(shape: Shape, C: int) -> int:
    return int(_native.lib().kvsel_out_tokens(shape.ref, int(C)))


def kvsel_score_path(shape: Shape, W: int, C: int = 0) -> int:
    return int(_native.lib().kvsel_score_path(shape.ref, int(W), int(C)))


def kvsel_window_logits(q_win, K, seq_offsets, W: int, logits=None, stream=None):
    """Raw window logits [layers, H, W, T] fp32 (diagnostic)."""
    K4, q4 = _as4(K), _as4(q_win)
    sh = shape_of(K, seq_offsets, q4.shape[2])
    _need(K4, "K"), _need(q4, "q_win", K4.dtype)
    L, H = K4.shape[0], q4.shape[2]
    if logits is None:
        logits = torch.empty((L, H, int(W), sh.T), dtype=torch.float32, device=K.device)
    _need(logits, "logits", torch.float32)
    _check(_native.lib().kvsel_window_logits(sh.ref, _ptr(q4), _ptr(K4), int(W), _ptr(logits),
                                             _stream(stream)), "kvsel_window_logits")
    return logits


def kvsel_score(q_win, K, seq_offsets, W: int, pool_kind: int, pool_k: int,
                votes=None, pooled=None, want_votes: bool = True, stream=None):
    """(votes, pooled), each [layers, H, T] fp32; votes is None if not wanted."""
    K4, q4 = _as4(K), _as4(q_win)
    sh = shape_of(K, seq_offsets, q4.shape[2])
    _need(K4, "K"), _need(q4, "q_win", K4.dtype)
    L, H = K4.shape[0], q4.shape[2]
    if votes is None and want_votes:
        votes = torch.empty((L, H, sh.T), dtype=torch.float32, device=K.device)
    if pooled is None:
        pooled = torch.empty((L, H, sh.T), dtype=torch.float32, device=K.device)
    for t, n in ((votes, "votes"), (pooled, "pooled")):
        if t is not None:
            _need(t, n, torch.float32)
    _check(_native.lib().kvsel_score(sh.ref, _ptr(q4), _ptr(K4), int(W), int(pool_kind),
                                     int(pool_k), _ptr(votes), _ptr(pooled), _stream(stream)),
           "kvsel_score")
    return votes, pooled


def kvsel_score_static(q_win, K, seq_offsets, W: int, pool_kind: int, pool_k: int,
                       votes=None, pooled=None, stream=None):
    """kvsel_score that allocates no device memory inside the library (its
    scratch is a fixed array in the library image); the output tensors are
    still the caller's."""
    K4, q4 = _as4(K), _as4(q_win)
    sh = shape_of(K, seq_offsets, q4.shape[2])
    _need(K4, "K"), _need(q4, "q_win", K4.dtype)
    L, H = K4.shape[0], q4.shape[2]
    if votes is None:
        votes = torch.empty((L, H, sh.T), dtype=torch.float32, device=K.device)
    if pooled is None:
        pooled = torch.empty((L, H, sh.T), dtype=torch.float32, device=K.device)
    _need(votes, "votes", torch.float32), _need(pooled, "pooled", torch.float32)
    _check(_native.lib().kvsel_score_static(sh.ref, _ptr(q4), _ptr(K4), int(W), int(pool_kind),
                                            int(pool_k), _ptr(votes), _ptr(pooled),
                                            _stream(stream)), "kvsel_score_static")
    return votes, pooled


def kvsel_score_static_bytes(shape: Shape, W: int) -> int:
    """Scratch bytes kvsel_score_static needs for this shape and window (-1: a
    rule is broken)."""
    return int(_native.lib().kvsel_score_static_bytes(shape.ref, int(W)))


def kvsel_select(pooled, seq_offsets, num_heads: int, W: int, C: int, out_idx=None,
                 stream=None):
    """out_idx [layers, T_out, H] int32 from pooled scores [layers, H, T]."""
    p3 = pooled if pooled.dim() == 3 else pooled.unsqueeze(0)
    _need(p3, "pooled", torch.float32)
    L = p3.shape[0]
    sh = Shape(L, num_heads, 1, KVSEL_F32, seq_offsets)
    t_out = kvsel_out_tokens(sh, C)
    if t_out < 0:
        raise KvselError(KVSEL_ERR_INVALID_ARG, "kvsel_select")
    if out_idx is None:
        out_idx = torch.empty((L, t_out, num_heads), dtype=torch.int32, device=pooled.device)
    _need(out_idx, "out_idx", torch.int32)
    _check(_native.lib().kvsel_select(sh.ref, _ptr(p3), int(W), int(C), _ptr(out_idx),
                                      _stream(stream)), "kvsel_select")
    return out_idx


def kvsel_compact(K, V, seq_offsets, out_idx, C: int, out_K=None, out_V=None, stream=None):
    """(out_K, out_V) [layers, T_out, H, D] gathered with out_idx [layers, T_out, H]
    (H may be a multiple of K's heads: output head h reads K/V head h / (H / H_kv))."""
    K4, V4 = _as4(K), _as4(V)
    H = out_idx.shape[-1]
    sh = shape_of(K, seq_offsets, H)
    _need(K4, "K"), _need(V4, "V", K4.dtype), _need(out_idx, "out_idx", torch.int32)
    L, D = K4.shape[0], K4.shape[3]
    t_out = kvsel_out_tokens(sh, C)
    if t_out < 0:
        raise KvselError(KVSEL_ERR_INVALID_ARG, "kvsel_compact")
    if out_K is None:
        out_K = torch.empty((L, t_out, H, D), dtype=K.dtype, device=K.device)
    if out_V is None:
        out_V = torch.empty((L, t_out, H, D), dtype=K.dtype, device=K.device)
    _need(out_K, "out_K", K4.dtype), _need(out_V, "out_V", K4.dtype)
    _check(_native.lib().kvsel_compact(sh.ref, _ptr(K4), _ptr(V4), _ptr(out_idx), int(C),
                                       _ptr(out_K), _ptr(out_V), _stream(stream)),
           "kvsel_compact")
    return out_K, out_V


def kvsel_snapkv(q_win, K, V, seq_offsets, W: int, C: int, pool_kind: int, pool_k: int,
                 out_idx=None, out_K=None, out_V=None, stream=None
                 ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """The fused path: (out_idx, out_K, out_V), over q_win's heads (with fewer
    K/V heads, query head h reads K/V head h / (H / H_kv): the expanded reading)."""
    K4, V4, q4 = _as4(K), _as4(V), _as4(q_win)
    sh = shape_of(K, seq_offsets, q4.shape[2])
    _need(K4, "K"), _need(V4, "V", K4.dtype), _need(q4, "q_win", K4.dtype)
    L, H, D = K4.shape[0], q4.shape[2], K4.shape[3]
    t_out = kvsel_out_tokens(sh, C)
    if t_out < 0:
        raise KvselError(KVSEL_ERR_INVALID_ARG, "kvsel_snapkv")
    dev = K.device
    if out_idx is None:
        out_idx = torch.empty((L, t_out, H), dtype=torch.int32, device=dev)
    if out_K is None:
        out_K = torch.empty((L, t_out, H, D), dtype=K.dtype, device=dev)
    if out_V is None:
        out_V = torch.empty((L, t_out, H, D), dtype=K.dtype, device=dev)
    _need(out_idx, "out_idx", torch.int32)
    _need(out_K, "out_K", K4.dtype), _need(out_V, "out_V", K4.dtype)
    _check(_native.lib().kvsel_snapkv(sh.ref, _ptr(q4), _ptr(K4), _ptr(V4), int(W), int(C),
                                      int(pool_kind), int(pool_k), _ptr(out_idx), _ptr(out_K),
                                      _ptr(out_V), _stream(stream)), "kvsel_snapkv")
    return out_idx, out_K, out_V


def kvsel_snapkv_grouped(q_win, K, V, seq_offsets, W: int, C: int, pool_kind: int,
                         pool_k: int, out_idx=None, out_K=None, out_V=None, stream=None
                         ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Group-shared selection (one per K/V head, votes of its query heads summed):
    (out_idx [layers, T_out, H_kv], out_K, out_V [layers, T_out, H_kv, D])."""
    K4, V4, q4 = _as4(K), _as4(V), _as4(q_win)
    sh = shape_of(K, seq_offsets, q4.shape[2])
    _need(K4, "K"), _need(V4, "V", K4.dtype), _need(q4, "q_win", K4.dtype)
    L, Hkv, D = K4.shape[0], K4.shape[2], K4.shape[3]
    t_out = kvsel_out_tokens(sh, C)
    if t_out < 0:
        raise KvselError(KVSEL_ERR_INVALID_ARG, "kvsel_snapkv_grouped")
    dev = K.device
    if out_idx is None:
        out_idx = torch.empty((L, t_out, Hkv), dtype=torch.int32, device=dev)
    if out_K is None:
        out_K = torch.empty((L, t_out, Hkv, D), dtype=K.dtype, device=dev)
    if out_V is None:
        out_V = torch.empty((L, t_out, Hkv, D), dtype=K.dtype, device=dev)
    _need(out_idx, "out_idx", torch.int32)
    _need(out_K, "out_K", K4.dtype), _need(out_V, "out_V", K4.dtype)
    _check(_native.lib().kvsel_snapkv_grouped(sh.ref, _ptr(q4), _ptr(K4), _ptr(V4), int(W),
                                              int(C), int(pool_kind), int(pool_k),
                                              _ptr(out_idx), _ptr(out_K), _ptr(out_V),
                                              _stream(stream)), "kvsel_snapkv_grouped")
    return out_idx, out_K, out_V


def kvsel_jacap_score(q_win, K, V, seq_offsets, W: int, tau: float = 10.0, beta: float = 0.9,
                      eps: float = 1e-6, scores=None, stream=None):
    """Jacap leverage scores [layers, H, T] fp32 (prefix positions; 0 elsewhere)."""
    K4, V4, q4 = _as4(K), _as4(V), _as4(q_win)
    sh = shape_of(K, seq_offsets, q4.shape[2])
    _need(K4, "K"), _need(V4, "V", K4.dtype), _need(q4, "q_win", K4.dtype)
    L, H = K4.shape[0], q4.shape[2]
    if scores is None:
        scores = torch.empty((L, H, sh.T), dtype=torch.float32, device=K.device)
    _need(scores, "scores", torch.float32)
    _check(_native.lib().kvsel_jacap_score(sh.ref, _ptr(q4), _ptr(K4), _ptr(V4), int(W),
                                           float(tau), float(beta), float(eps), _ptr(scores),
                                           _stream(stream)), "kvsel_jacap_score")
    return scores


def kvsel_jacap(q_win, K, V, seq_offsets, W: int, C: int, tau: float = 10.0, beta: float = 0.9,
                eps: float = 1e-6, out_idx=None, out_K=None, out_V=None, stream=None):
    """Jacap selection: (out_idx, out_K, out_V) with kvsel_snapkv's layouts."""
    K4, V4, q4 = _as4(K), _as4(V), _as4(q_win)
    sh = shape_of(K, seq_offsets, q4.shape[2])
    _need(K4, "K"), _need(V4, "V", K4.dtype), _need(q4, "q_win", K4.dtype)
    L, H, D = K4.shape[0], q4.shape[2], K4.shape[3]
    t_out = kvsel_out_tokens(sh, C)
    if t_out < 0:
        raise KvselError(KVSEL_ERR_INVALID_ARG, "kvsel_jacap")
    dev = K.device
    if out_idx is None:
        out_idx = torch.empty((L, t_out, H), dtype=torch.int32, device=dev)
    if out_K is None:
        out_K = torch.empty((L, t_out, H, D), dtype=K.dtype, device=dev)
    if out_V is None:
        out_V = torch.empty((L, t_out, H, D), dtype=K.dtype, device=dev)
    _check(_native.lib().kvsel_jacap(sh.ref, _ptr(q4), _ptr(K4), _ptr(V4), int(W), int(C),
                                     float(tau), float(beta), float(eps), _ptr(out_idx),
                                     _ptr(out_K), _ptr(out_V), _stream(stream)), "kvsel_jacap")
    return out_idx, out_K, out_V


def kvsel_snapkv_host(q_win, K, V, seq_offsets, W: int, C: int, pool_kind: int, pool_k: int,
                      out_idx=None, out_K=None, out_V=None, stream=None):
    """kvsel_snapkv on CPU tensors (V and the outputs pinned): (out_idx, out_K, out_V)
    pinned CPU tensors, complete once `stream` reaches the point after the call."""
    K4, V4, q4 = _as4(K), _as4(V), _as4(q_win)
    for t, n in ((K4, "K"), (V4, "V"), (q4, "q_win")):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous CPU tensor")
    if not V4.is_pinned():
        raise ValueError("V must be pinned (page-locked) host memory")
    if K4.dtype not in _DTYPES or V4.dtype != K4.dtype or q4.dtype != K4.dtype:
        raise ValueError("q_win, K and V must share a dtype, bf16 or fp32")
    sh = shape_of(K, seq_offsets, q4.shape[2])
    L, H, D = K4.shape[0], q4.shape[2], K4.shape[3]
    t_out = kvsel_out_tokens(sh, C)
    if t_out < 0:
        raise KvselError(KVSEL_ERR_INVALID_ARG, "kvsel_snapkv_host")
    if out_idx is None:
        out_idx = torch.empty((L, t_out, H), dtype=torch.int32, pin_memory=True)
    if out_K is None:
        out_K = torch.empty((L, t_out, H, D), dtype=K.dtype, pin_memory=True)
    if out_V is None:
        out_V = torch.empty((L, t_out, H, D), dtype=K.dtype, pin_memory=True)
    for t, n in ((out_idx, "out_idx"), (out_K, "out_K"), (out_V, "out_V")):
        if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous pinned CPU tensor")
    _check(_native.lib().kvsel_snapkv_host(sh.ref, _ptr(q4), _ptr(K4), _ptr(V4), int(W), int(C),
                                           int(pool_kind), int(pool_k), _ptr(out_idx),
                                           _ptr(out_K), _ptr(out_V), _stream(stream)),
           "kvsel_snapkv_host")
    return out_idx, out_K, out_V


def kvsel_decode_attention(q, K, V, cache_offsets, K_new=None, V_new=None, g: int = 0,
                           out=None, lse=None, want_lse: bool = True, stream=None):
    """(out [layers, S, H, D] fp32, lse [layers, S, H] fp32 or None): one query per
    (layer, sequence, query head) over its cache rows (packed by cache_offsets)
    and then its g appended rows. q [layers, S, H, D]; K, V [layers, T, H_kv, D];
    K_new, V_new [layers, S * g, H_kv, D]."""
    q4, K4, V4 = q if q.dim() == 4 else q.unsqueeze(0), _as4(K), _as4(V)
    L, S, H, D = q4.shape
    if len(cache_offsets) != S + 1:
        raise ValueError("cache_offsets must have num_seqs + 1 entries")
    _need(K4, "K"), _need(V4, "V", K4.dtype), _need(q4, "q", K4.dtype)
    sh = Shape(L, H, D, _DTYPES[K4.dtype], cache_offsets, num_kv_heads=K4.shape[2])
    kn = vn = None
    if g:
        kn, vn = _as4(K_new), _as4(V_new)
        _need(kn, "K_new", K4.dtype), _need(vn, "V_new", K4.dtype)
    if out is None:
        out = torch.empty((L, S, H, D), dtype=torch.float32, device=K.device)
    if lse is None and want_lse:
        lse = torch.empty((L, S, H), dtype=torch.float32, device=K.device)
    _need(out, "out", torch.float32)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    _check(_native.lib().kvsel_decode_attention(sh.ref, _ptr(q4), _ptr(K4), _ptr(V4), int(g),
                                                _ptr(kn), _ptr(vn), _ptr(out), _ptr(lse),
                                                _stream(stream)), "kvsel_decode_attention")
    return out, lse


def kvsel_reverse_attention(Q, K, V, seq_offsets, positions=None, out=None, lse=None,
                            want_lse: bool = True, stream=None):
    """(out [layers, T, H, D] fp32, lse [layers, H, T] fp32 or None): every row
    i of a sequence attends to the rows of its sequence at later positions
    only (positions [T] int32 sequence-relative, default the row order); a row
    with no later row gets out = 0, lse = -inf. Q [layers, T, H, D]; K, V
    [layers, T, H_kv, D]; bf16, D = 128."""
    Q4, K4, V4 = _as4(Q), _as4(K), _as4(V)
    L, T, H, D = Q4.shape
    _need(K4, "K"), _need(V4, "V", K4.dtype), _need(Q4, "Q", K4.dtype)
    sh = Shape(L, H, D, _DTYPES[K4.dtype], seq_offsets, num_kv_heads=K4.shape[2])
    if positions is not None:
        _need(positions, "positions", torch.int32)
    if out is None:
        out = torch.empty((L, T, H, D), dtype=torch.float32, device=K.device)
    if lse is None and want_lse:
        lse = torch.empty((L, H, T), dtype=torch.float32, device=K.device)
    _need(out, "out", torch.float32)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    _check(_native.lib().kvsel_reverse_attention(sh.ref, _ptr(Q4), _ptr(K4), _ptr(V4),
                                                 _ptr(positions), _ptr(out), _ptr(lse),
                                                 _stream(stream)), "kvsel_reverse_attention")
    return out, lse


def kvsel_decode_quality(lse_keep, lse_full, out_keep, out_full, mass=None, err=None,
                         stream=None):
    """(mass, err), each shaped like lse: exp(lse_keep - lse_full) and
    ||out_full - out_keep||_2 over the last dimension of out."""
    n = lse_keep.numel()
    D = out_keep.shape[-1]
    for t, nm in ((lse_keep, "lse_keep"), (lse_full, "lse_full"), (out_keep, "out_keep"),
                  (out_full, "out_full")):
        _need(t, nm, torch.float32)
    if mass is None:
        mass = torch.empty_like(lse_keep)
    if err is None:
        err = torch.empty_like(lse_keep)
    _check(_native.lib().kvsel_decode_quality(int(n), int(D), _ptr(lse_keep), _ptr(lse_full),
                                              _ptr(out_keep), _ptr(out_full), _ptr(mass),
                                              _ptr(err), _stream(stream)),
           "kvsel_decode_quality")
    return mass, err


def kvsel_cache_lengths(seq_offsets, C: int, g: int):
    """(physical_length, next_logical): per sequence min(L_b, C) + g and L_b + g."""
    sh = Shape(1, 1, 1, KVSEL_BF16, seq_offsets)
    n = max(0, len(seq_offsets) - 1)
    phys = (ctypes.c_int64 * max(1, n))()
    logi = (ctypes.c_int64 * max(1, n))()
    _check(_native.lib().kvsel_cache_lengths(sh.ref, int(C), int(g), phys, logi),
           "kvsel_cache_lengths")
    return [phys[i] for i in range(n)], [logi[i] for i in range(n)]


def kvsel_device_status(stream=None) -> int:
    return int(_native.lib().kvsel_device_status(_stream(stream)))


def kvsel_set_wait_limit_ns(ns: int) -> None:
    _check(_native.lib().kvsel_set_wait_limit_ns(int(ns)), "kvsel_set_wait_limit_ns")


def kvsel_debug_inject(what: int) -> None:
    _check(_native.lib().kvsel_debug_inject(int(what)), "kvsel_debug_inject")


def kvsel_profile_begin(max_calls: int) -> None:
    _check(_native.lib().kvsel_profile_begin(int(max_calls)), "kvsel_profile_begin")


def kvsel_profile_end():
    """(summed ms per stage [score, select, gather], number of recorded calls)."""
    ms = (ctypes.c_double * 3)()
    calls = ctypes.c_int32(0)
    _check(_native.lib().kvsel_profile_end(ms, ctypes.byref(calls)), "kvsel_profile_end")
    return [ms[0], ms[1], ms[2]], calls.value


def kvsel_release() -> None:
    _native.lib().kvsel_release()


def kvsel_workspace_bytes() -> int:
    """Bytes of the library's cudaMalloc'd workspace held on the current device."""
    return int(_native.lib().kvsel_workspace_bytes())
