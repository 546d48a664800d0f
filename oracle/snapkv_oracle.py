"""SnapKV observation-window KV selection: plain, slow, fp64 CPU oracle.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its ``cpu_baseline`` leg and ``--impl reference``) may import,
call or execute this module. The CUDA library never links it and shares no
code, table or constant with it.

Source: the page "SnapKV: choosing the KV cache of a long prompt with an
observation window" (SnapKV：用观察窗口为长提示词选择 KV Cache,
charlestar.github.io, 2026-10-20). Section names used below:

* [Partition]  "要缩小的是提示词缓存，不是忘记位置的来源": prompt length L,
  window W = last W tokens, prefix P = L - W, budget C keeps the whole window
  plus C - W prefix positions; selection is per layer and per head.
* [Votes]      "投票必须来自完整提示词的因果 softmax": logits of the W window
  queries against all L keys scaled by 1/sqrt(D), causal mask j <= t, softmax
  denominator over every visible position (prefix AND window columns), then
  votes s_j = sum over the W rows of the prefix-column probabilities.
* [Pooling]    "池化把一个峰值扩展成邻域偏好": odd width, stride 1, zero padding;
  the average divides by the full width even at the edges; max pooling is the
  alternative; then the C - W prefix positions with the highest pooled score
  are kept and the whole window is appended.
* [Example]    "从 Q 和 K 开始算一次完整选择": the L=8, W=2, C=5, D=2 worked
  example, argument rules, the short-prompt bypass (L < C keeps everything),
  the non-finite-dot-product error, and the (-score, index) order that breaks
  ties towards the smaller index.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(worked example, counterexample, closed forms, invariants, brute force).

Each step is a separate module-level function, looked up at call time by
``snapkv_head``, so tests can swap one step for a deliberately wrong variant
and check that the pins catch it.
"""

from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np

POOLINGS = ("avg", "max")


class OracleArgumentError(ValueError):
    """Raised where the page's reference function raises ValueError."""


# ---------------------------------------------------------------------------
# Argument rules ([Example]: the rules its CPU function checks before work)
# ---------------------------------------------------------------------------

def _is_int(x) -> bool:
    return isinstance(x, (int, np.integer)) and not isinstance(x, (bool, np.bool_))


def check_head_args(q_win, keys, values, capacity, kernel_size, pooling):
    """Validate one head's inputs with the page's rules.

    q_win: (W, D) window queries (rows t = P..L-1); keys, values: (L, D).
    Rules: nonempty prompt, K and V of equal length, positive head dim,
    equal row widths, finite numbers, positive integer window / capacity /
    kernel, W <= L, C > W, odd kernel, pooling in {avg, max}.
    """
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    q_win = np.asarray(q_win, dtype=np.float64)
    if keys.ndim != 2 or keys.shape[0] == 0:
        raise OracleArgumentError("K must be a nonempty (L, D) matrix")
    if values.shape[0] != keys.shape[0]:
        raise OracleArgumentError("K and V need the same prompt length")
    if keys.shape[1] == 0:
        raise OracleArgumentError("head dimension must be positive")
    if q_win.ndim != 2 or values.ndim != 2 or \
            q_win.shape[1] != keys.shape[1] or values.shape[1] != keys.shape[1]:
        raise OracleArgumentError("all head vectors need the same dimension")
    for t in (q_win, keys, values):
        if not np.isfinite(t).all():
            raise OracleArgumentError("inputs must be finite")
    window = q_win.shape[0]
    for n in (window, capacity, kernel_size):
        if not _is_int(n) or n <= 0:
            raise OracleArgumentError("window, capacity and kernel must be positive integers")
    if window > keys.shape[0] or capacity <= window:
        raise OracleArgumentError("need W <= L and C > W")
    if kernel_size % 2 != 1 or pooling not in POOLINGS:
        raise OracleArgumentError("need an odd kernel and avg or max pooling")
    return q_win, keys, values


# ---------------------------------------------------------------------------
# The steps ([Votes], [Pooling])
# ---------------------------------------------------------------------------

def window_logits(q_win: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """z[r, j] = q_{P+r} . k_j / sqrt(D) for every key j in [0, L).

    Returns a (W, L) fp64 matrix; masking happens in causal_probabilities.
    """
    d = keys.shape[1]
    return (q_win @ keys.T) / math.sqrt(d)


def causal_probabilities(z: np.ndarray) -> np.ndarray:
    """Row r is window query t = P + r; it sees keys j <= t.

    p[r, j] = exp(z[r, j] - m_r) / sum_{i <= t} exp(z[r, i] - m_r) for j <= t
    and 0 for j > t, with m_r the largest visible logit. The denominator runs
    over every visible column, window columns included.
    """
    w, l = z.shape
    p_len = l - w
    p = np.zeros_like(z)
    for r in range(w):
        t = p_len + r
        visible = z[r, : t + 1]
        m = visible.max()
        e = np.exp(visible - m)
        p[r, : t + 1] = e / e.sum()
    return p


def prefix_votes(p: np.ndarray) -> np.ndarray:
    """s_j = sum over the W window rows of p[r, j], for prefix columns j < P."""
    w, l = p.shape
    return p[:, : l - w].sum(axis=0)


def pool_scores(s: np.ndarray, kernel_size: int, pooling: str) -> np.ndarray:
    """1-D pooling of the prefix votes: width k (odd), stride 1, zero padding.

    avg: (sum of the in-range neighbours j-R..j+R) / k, the divisor staying k
         at the edges (out-of-range neighbours count as zeros);
    max: the largest in-range neighbour (votes are >= 0, so this equals a
         zero-padded max).
    Only prefix votes are neighbours: the window is not part of the array.
    """
    p_len = s.shape[0]
    radius = kernel_size // 2
    if pooling == "avg":
        acc = np.zeros(p_len, dtype=np.float64)
    else:
        acc = np.full(p_len, -np.inf, dtype=np.float64)
    for d in range(-radius, radius + 1):
        # neighbour index i = j + d is in range for j in [lo, hi)
        lo, hi = max(0, -d), min(p_len, p_len - d)
        if lo >= hi:
            continue
        if pooling == "avg":
            acc[lo:hi] += s[lo + d: hi + d]
        else:
            acc[lo:hi] = np.maximum(acc[lo:hi], s[lo + d: hi + d])
    if pooling == "avg":
        return acc / kernel_size
    return acc


def top_prefix(pooled: np.ndarray, n_keep: int) -> List[int]:
    """The n_keep prefix positions first in the order key (-pooled_j, j).

    Returned in that order: highest score first, equal scores by smaller index.
    """
    p_len = pooled.shape[0]
    order = np.lexsort((np.arange(p_len), -np.asarray(pooled, dtype=np.float64)))
    return [int(j) for j in order[:n_keep]]


def window_row_exp_sums(q_win: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """Unshifted row sums sum_{j <= t} exp(z[r, j]) (the worked example prints them)."""
    z = window_logits(np.asarray(q_win, np.float64), np.asarray(keys, np.float64))
    w, l = z.shape
    return np.array([np.exp(z[r, : l - w + r + 1]).sum() for r in range(w)])


# ---------------------------------------------------------------------------
# One head ([Partition], [Example])
# ---------------------------------------------------------------------------

def snapkv_head(q_win, keys, values, capacity: int, kernel_size: int = 3,
                pooling: str = "avg") -> Dict[str, object]:
    """Select and gather one (layer, head)'s prompt cache.

    Returns indices (selected prefix in (-pooled, j) order, then the window in
    ascending order; or 0..L-1 when L < C), the gathered keys and values (same
    indices for both), and the intermediate votes, pooled scores and
    probabilities (empty for the bypass).
    """
    q_win, keys, values = check_head_args(q_win, keys, values, capacity,
                                          kernel_size, pooling)
    length, window = keys.shape[0], q_win.shape[0]
    if length < capacity:
        idx = list(range(length))
        return {"indices": idx, "keys": keys.copy(), "values": values.copy(),
                "votes": np.zeros(0), "pooled": np.zeros(0), "probs": None}
    z = window_logits(q_win, keys)
    if not np.isfinite(z).all():
        raise OracleArgumentError("non-finite dot product")
    p = causal_probabilities(z)
    s = prefix_votes(p)
    pooled = pool_scores(s, kernel_size, pooling)
    prefix = length - window
    idx = top_prefix(pooled, capacity - window) + list(range(prefix, length))
    return {"indices": idx, "keys": keys[idx], "values": values[idx],
            "votes": s, "pooled": pooled, "probs": p}


def select_from_pooled(pooled_prefix: np.ndarray, length: int, window: int,
                       capacity: int) -> List[int]:
    """Selection alone, from given pooled prefix scores (the select stage).

    L < C: identity. Otherwise top (C - W) prefix positions by (-score, j),
    then the window P..L-1.
    """
    if length < capacity:
        return list(range(length))
    prefix = length - window
    pooled_prefix = np.asarray(pooled_prefix, dtype=np.float64)
    assert pooled_prefix.shape[0] == prefix
    return top_prefix(pooled_prefix, capacity - window) + list(range(prefix, length))


# ---------------------------------------------------------------------------
# Packed multi-layer, multi-head, ragged batches (each (layer, seq, head) is
# an independent instance: [Partition] "selection happens per layer and head")
# ---------------------------------------------------------------------------

def snapkv_packed(q_win: np.ndarray, keys: np.ndarray, values: np.ndarray,
                  seq_offsets: Sequence[int], window: int, capacity: int,
                  kernel_size: int, pooling: str,
                  heads: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
    """Run snapkv_head over every (layer, sequence, head) of a packed batch.

    Layouts: q_win (layers, S*W, H, D); keys, values (layers, T, H, D) with
    sequence b at tokens seq_offsets[b]..seq_offsets[b+1]-1. Outputs:
    out_idx (layers, T_out, H) int64 positions within the sequence, out_K,
    out_V (layers, T_out, H, D), votes and pooled (layers, H, T) with zeros at
    window and bypass positions; T_out = sum_b min(L_b, C).
    ``heads`` restricts the work to some heads (other outputs stay zero).
    """
    q_win = np.asarray(q_win, np.float64)
    keys = np.asarray(keys, np.float64)
    values = np.asarray(values, np.float64)
    n_layers, total, n_heads, dim = keys.shape
    offs = [int(x) for x in seq_offsets]
    lens = [offs[b + 1] - offs[b] for b in range(len(offs) - 1)]
    kept = [min(l, capacity) for l in lens]
    out_offs = np.concatenate([[0], np.cumsum(kept)]).astype(int)
    t_out = int(out_offs[-1])
    out_idx = np.zeros((n_layers, t_out, n_heads), np.int64)
    out_k = np.zeros((n_layers, t_out, n_heads, dim))
    out_v = np.zeros((n_layers, t_out, n_heads, dim))
    votes = np.zeros((n_layers, n_heads, total))
    pooled = np.zeros((n_layers, n_heads, total))
    head_list = range(n_heads) if heads is None else heads
    for layer in range(n_layers):
        for b, length in enumerate(lens):
            o, oo = offs[b], out_offs[b]
            for h in head_list:
                res = snapkv_head(q_win[layer, b * window:(b + 1) * window, h],
                                  keys[layer, o:o + length, h],
                                  values[layer, o:o + length, h],
                                  capacity, kernel_size, pooling)
                n = len(res["indices"])
                out_idx[layer, oo:oo + n, h] = res["indices"]
                out_k[layer, oo:oo + n, h] = res["keys"]
                out_v[layer, oo:oo + n, h] = res["values"]
                pl = len(res["votes"])
                votes[layer, h, o:o + pl] = res["votes"]
                pooled[layer, h, o:o + pl] = res["pooled"]
    return {"out_idx": out_idx, "out_K": out_k, "out_V": out_v,
            "votes": votes, "pooled": pooled, "out_offsets": out_offs}
