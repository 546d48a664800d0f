"""Reverse-mask attention of the counter-causal scorer: plain fp64 CPU oracle.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` may import it; the CUDA library
shares nothing with it.

Source: the page "来自未来的信号：用反因果惊奇度做 KV Cache 淘汰" (signals from
the future: KV-cache eviction by counter-causal surprise, zhongzhuzhou.org,
2026-08-01):

* section 3.2 (the approximation that reuses the cached K/V under a reversed
  mask), step 1: the sequence keeps its order and its position ids, and the
  causal mask is replaced by a strictly upper-triangular one, so position i
  attends only to positions j > i; step 3: the keys and values are the cached
  ones (already rotated at their original positions), only the queries are
  recomputed at the original positions; step 5: the last position has no
  future context and is given the largest surprise;
* section 4, Algorithm 3 (one memory refresh): every one of the J + h cached
  candidates is scored, then the memory is reordered by surprise, so cache
  slots need not follow position order.

Readings (ours, where the page leaves it open): the attention is scaled
dot-product attention with the scale 1/sqrt(D) over the keys whose original
position is larger than the query's own; out_i = sum_j p_j v_j and lse_i is
the natural log of the softmax denominator sum_j exp(q_i . k_j / sqrt(D)); a
position with no later key (the last one) has out = 0 and lse = -inf (the
page assigns it the largest surprise, so no attention output is used);
positions default to the row order within the sequence; with grouped K/V
heads query head h reads K/V head h // (H / H_kv). The surprise itself (the
true token's logit through the model's output layer) needs model weights and
is not computed.

Parity status: pinned by ``tests/test_oracle_reverse.py`` (the decode
oracle on each query's future rows, a library attention with an explicit
strictly-upper mask, the equal-key closed form, the boundary rows, position
permutation, future-only dependence, planted mistakes).
"""

from __future__ import annotations

from typing import Dict, Optional, Sequence

import numpy as np

from .snapkv_oracle import OracleArgumentError


def reverse_attention(q, keys, values, positions: Optional[Sequence[int]] = None):
    """One head of one sequence: (out (n, Dv), lse (n,)).

    q, keys: (n, D); values: (n, Dv); positions: n distinct integers (the
    original position of each row), default 0 .. n-1.
    """
    q = np.asarray(q, np.float64)
    keys = np.asarray(keys, np.float64)
    values = np.asarray(values, np.float64)
    n = q.shape[0]
    if q.ndim != 2 or keys.shape != q.shape or values.shape[0] != n:
        raise OracleArgumentError("q, keys (n, D) and values (n, Dv)")
    pos = np.arange(n) if positions is None else np.asarray(positions, np.int64)
    if pos.shape != (n,) or len(set(pos.tolist())) != n:
        raise OracleArgumentError("positions: n distinct integers")
    scale = 1.0 / np.sqrt(q.shape[1])
    out = np.zeros((n, values.shape[1]))
    lse = np.full(n, -np.inf)
    for i in range(n):
        future = pos > pos[i]
        if not future.any():
            continue
        z = keys[future] @ q[i] * scale
        m = z.max()
        e = np.exp(z - m)
        out[i] = (e / e.sum()) @ values[future]
        lse[i] = m + np.log(e.sum())
    return out, lse


def reverse_packed(q, keys, values, offsets: Sequence[int],
                   positions: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
    """Every (layer, sequence, query head) of a packed batch.

    q (layers, T, H, D); keys, values (layers, T, H_kv, D), sequence b at rows
    offsets[b] .. offsets[b+1]-1; positions (T,) sequence-relative original
    positions (None: the row order). Returns out (layers, T, H, D) and lse
    (layers, H, T).
    """
    q = np.asarray(q, np.float64)
    keys = np.asarray(keys, np.float64)
    values = np.asarray(values, np.float64)
    n_layers, total, h_q, dim = q.shape
    h_kv = keys.shape[2]
    if h_q % h_kv:
        raise OracleArgumentError("query heads must be a multiple of key/value heads")
    group = h_q // h_kv
    offs = [int(x) for x in offsets]
    if offs[0] != 0 or offs[-1] != total or any(b < a for a, b in zip(offs, offs[1:])):
        raise OracleArgumentError("offsets: nondecreasing from 0 to T")
    out = np.zeros((n_layers, total, h_q, values.shape[3]))
    lse = np.full((n_layers, h_q, total), -np.inf)
    for layer in range(n_layers):
        for b in range(len(offs) - 1):
            rows = slice(offs[b], offs[b + 1])
            if offs[b + 1] == offs[b]:
                continue
            pb = None if positions is None else np.asarray(positions)[rows]
            for h in range(h_q):
                o, l = reverse_attention(q[layer, rows, h], keys[layer, rows, h // group],
                                         values[layer, rows, h // group], pb)
                out[layer, rows, h] = o
                lse[layer, h, rows] = l
    return {"out": out, "lse": lse}
