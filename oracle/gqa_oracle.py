"""Grouped-query (GQA) selection: plain, slow, fp64 CPU oracle.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` may import it; the CUDA library
shares nothing with it.

Source: the page "SnapKV: choosing the KV cache of a long prompt with an
observation window" (charlestar.github.io), section [GQA] "GQA 下的缓存节省不能
只算 C 除以 L" (with GQA the cache saving is not just C / L): H_kv key/value
heads serve H_q = G * H_kv query heads. The integration the page describes
expands K and V to the H_q query heads (repeat_kv) and then selects per query
head, so the kept cache is counted per query head. A selection shared by the
G query heads of one group, which would keep the native H_kv cache, is left
open by the page ("must be designed separately").

Readings (ours, where the page is open):

* ``repeat`` mode: query head h uses key/value head h // G; each query head
  is an ordinary instance ([Votes], [Pooling] of ``snapkv_oracle``); outputs
  have H_q heads. This equals expanding K and V with repeat_kv first.
* ``group`` mode: one selection per key/value head. Each of its G query heads
  computes its own causal-softmax votes against the shared keys (the W window
  rows of that head); the group's vote of prefix position j is the sum of the
  G heads' votes, in head order; pooling and the top-(C - W) selection by
  (-score, j) then run once on that sum, and K and V are gathered once. The
  bypass (L < C keeps everything) is unchanged. Outputs have H_kv heads.

Parity status: pinned by ``tests/test_oracle_gqa.py`` (expansion identity,
G = 1 reduction, identical heads, uniform closed form, brute force).
"""

from __future__ import annotations

from typing import Dict, Sequence

import numpy as np

from . import snapkv_oracle as so


def snapkv_group(q_group, keys, values, capacity: int, kernel_size: int = 3,
                 pooling: str = "avg") -> Dict[str, object]:
    """Group-shared selection for one (layer, key/value head).

    q_group: (G, W, D) window queries of the group's G query heads; keys,
    values: (L, D). Returns indices (selected prefix in (-pooled, j) order,
    then the window ascending; 0..L-1 when L < C), the gathered keys and
    values, the summed votes, the pooled scores and each head's votes.
    """
    q_group = np.asarray(q_group, dtype=np.float64)
    if q_group.ndim != 3 or q_group.shape[0] < 1:
        raise so.OracleArgumentError("q_group must be (G, W, D) with G >= 1")
    checked = [so.check_head_args(q_group[g], keys, values, capacity, kernel_size, pooling)
               for g in range(q_group.shape[0])]
    keys, values = checked[0][1], checked[0][2]
    length, window = keys.shape[0], q_group.shape[1]
    if length < capacity:
        return {"indices": list(range(length)), "keys": keys.copy(),
                "values": values.copy(), "votes": np.zeros(0), "pooled": np.zeros(0),
                "head_votes": []}
    head_votes = []
    for g in range(q_group.shape[0]):
        z = so.window_logits(checked[g][0], keys)
        if not np.isfinite(z).all():
            raise so.OracleArgumentError("non-finite dot product")
        head_votes.append(so.prefix_votes(so.causal_probabilities(z)))
    votes = np.zeros_like(head_votes[0])
    for s in head_votes:          # head order
        votes = votes + s
    pooled = so.pool_scores(votes, kernel_size, pooling)
    prefix = length - window
    idx = so.top_prefix(pooled, capacity - window) + list(range(prefix, length))
    return {"indices": idx, "keys": keys[idx], "values": values[idx],
            "votes": votes, "pooled": pooled, "head_votes": head_votes}


def snapkv_packed_gqa(q_win: np.ndarray, keys: np.ndarray, values: np.ndarray,
                      seq_offsets: Sequence[int], window: int, capacity: int,
                      kernel_size: int, pooling: str, mode: str) -> Dict[str, np.ndarray]:
    """Every (layer, sequence, head) of a packed GQA batch.

    Layouts: q_win (layers, S*W, H_q, D); keys, values (layers, T, H_kv, D),
    H_q = G * H_kv. ``mode`` "repeat": outputs over the H_q query heads (query
    head h reads key/value head h // G); "group": outputs over the H_kv heads.
    out_idx (layers, T_out, heads) positions within the sequence, out_K and
    out_V (layers, T_out, heads, D); votes and pooled (layers, heads, T),
    zero at window and bypass positions (group: the summed votes).
    """
    if mode not in ("repeat", "group"):
        raise so.OracleArgumentError("mode must be 'repeat' or 'group'")
    q_win = np.asarray(q_win, np.float64)
    keys = np.asarray(keys, np.float64)
    values = np.asarray(values, np.float64)
    n_layers, total, h_kv, dim = keys.shape
    h_q = q_win.shape[2]
    if h_q % h_kv:
        raise so.OracleArgumentError("query heads must be a multiple of key/value heads")
    group = h_q // h_kv
    n_heads = h_q if mode == "repeat" else h_kv
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
    for layer in range(n_layers):
        for b, length in enumerate(lens):
            o, oo = offs[b], out_offs[b]
            qs = q_win[layer, b * window:(b + 1) * window]
            for h in range(n_heads):
                if mode == "repeat":
                    kvh = h // group
                    res = so.snapkv_head(qs[:, h], keys[layer, o:o + length, kvh],
                                         values[layer, o:o + length, kvh],
                                         capacity, kernel_size, pooling)
                else:
                    q_group = np.stack([qs[:, h * group + g] for g in range(group)])
                    res = snapkv_group(q_group, keys[layer, o:o + length, h],
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
