"""Decode-side consumer of a compacted cache: plain fp64 CPU oracle.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` may import it; the CUDA library
shares nothing with it.

Source: the page "SnapKV: choosing the KV cache of a long prompt with an
observation window" (charlestar.github.io):

* section [Deletion] "删除位置为什么会改变输出" (why deleting positions changes
  the output): fix one future query; alpha_j are its attention probabilities
  over the full cache; S is the kept set and m = sum_{j in S} alpha_j the
  probability mass the full softmax gives it. Attention over S alone
  re-normalises the kept weights to alpha_j / m. With O_keep and O_drop the
  internally normalised value sums of the kept and the dropped positions,
  O_full = m O_keep + (1 - m) O_drop, so O_full - O_keep = (1 - m)(O_drop -
  O_keep), whose norm is at most 2 (1 - m) V_max when every ||V_j|| <= V_max.
  Its example: two equal logits with V = [0, 10] give 5 in full and 0 once
  only the first position is kept.
* section [Prefill] "当前 prefill 仍读完整 K/V，压缩缓存服务后续 decode": once g
  generated tokens have had their K/V appended, the cache holds min(L, C) + g
  rows.
* section [Positions] "缓存槽位不能代替 RoPE 的原始位置": kept keys keep their
  original (already encoded) positions; the next token's logical position is
  L + g while its physical slot is min(L, C) + g.
* section [Example], last paragraph: a single query reading the whole kept
  history is unchanged when K and V rows are permuted together.

Readings (ours): the future query attends, unmasked, to every row of the cache
(all of them are in its past), with the scale 1/sqrt(D) of the scoring; the
g appended rows are in both the full and the compacted cache, so S is the kept
prompt positions plus the appended ones; lse is the natural logarithm of the
sum of exp(q . k / sqrt(D)) over the attended rows.

Parity status: pinned by ``tests/test_oracle_decode.py`` (the page's example,
the decomposition identity and bound, permutation invariance, equal-key
closed form, the page's position table).
"""

from __future__ import annotations

from typing import Dict, Sequence, Tuple

import numpy as np

from .snapkv_oracle import OracleArgumentError


def decode_attention(q, keys, values) -> Tuple[np.ndarray, float]:
    """One query over a set of cache rows: (output, lse).

    q: (D,); keys: (n, D); values: (n, Dv). output = sum_j p_j values_j with
    p = softmax(keys q / sqrt(D)); lse = log sum_j exp(keys_j . q / sqrt(D)).
    """
    q = np.asarray(q, np.float64)
    keys = np.asarray(keys, np.float64)
    values = np.asarray(values, np.float64)
    if keys.ndim != 2 or keys.shape[0] < 1 or keys.shape[1] != q.shape[0]:
        raise OracleArgumentError("keys must be (n >= 1, D) with D = len(q)")
    if values.shape[0] != keys.shape[0]:
        raise OracleArgumentError("values must have one row per key")
    z = keys @ q / np.sqrt(q.shape[0])
    zmax = z.max()
    e = np.exp(z - zmax)
    total = e.sum()
    return (e / total) @ values, float(zmax + np.log(total))


def full_probabilities(q, keys) -> np.ndarray:
    """alpha_j: the query's softmax over every row of the full cache."""
    q = np.asarray(q, np.float64)
    z = np.asarray(keys, np.float64) @ q / np.sqrt(q.shape[0])
    e = np.exp(z - z.max())
    return e / e.sum()


def decompose(q, keys, values, kept: Sequence[int]) -> Dict[str, object]:
    """The [Deletion] quantities for one query, full cache keys/values and a
    kept row set: alpha, m, O_full, O_keep (attention over the kept rows
    alone), O_drop (over the dropped rows alone; None when nothing is
    dropped) and the error ||O_full - O_keep||_2."""
    keys = np.asarray(keys, np.float64)
    values = np.asarray(values, np.float64)
    kept = sorted(set(int(j) for j in kept))
    if not kept:
        raise OracleArgumentError("the kept set must not be empty")
    dropped = [j for j in range(keys.shape[0]) if j not in set(kept)]
    alpha = full_probabilities(q, keys)
    out_full, _ = decode_attention(q, keys, values)
    out_keep, _ = decode_attention(q, keys[kept], values[kept])
    out_drop = decode_attention(q, keys[dropped], values[dropped])[0] if dropped else None
    m = float(alpha[kept].sum())
    return {"alpha": alpha, "m": m, "out_full": out_full, "out_keep": out_keep,
            "out_drop": out_drop, "err": float(np.linalg.norm(out_full - out_keep))}


def cache_lengths(length: int, capacity: int, generated: int) -> Dict[str, int]:
    """[Prefill] / [Positions] bookkeeping after `generated` appended tokens:
    the physical cache length (also the next write slot) and the next
    logical position."""
    if length < 0 or capacity < 1 or generated < 0:
        raise OracleArgumentError("length >= 0, capacity >= 1, generated >= 0")
    phys = min(length, capacity) + generated
    return {"physical_length": phys, "next_slot": phys, "next_logical": length + generated}


def decode_packed(q, keys, values, cache_offsets: Sequence[int], k_new=None, v_new=None,
                  generated: int = 0) -> Dict[str, np.ndarray]:
    """Every (layer, sequence, query head) of a packed batch.

    q (layers, S, H, D); keys, values (layers, T, H_kv, D) packed by
    cache_offsets (S + 1 entries); k_new, v_new (layers, S * g, H_kv, D): the
    g appended rows of sequence b at rows b*g .. b*g + g - 1 (None when g = 0).
    Query head h reads key/value head h // (H / H_kv). Returns out (layers, S,
    H, D) and lse (layers, S, H).
    """
    q = np.asarray(q, np.float64)
    keys = np.asarray(keys, np.float64)
    values = np.asarray(values, np.float64)
    n_layers, n_seqs, h_q, dim = q.shape
    h_kv = keys.shape[2]
    if h_q % h_kv:
        raise OracleArgumentError("query heads must be a multiple of key/value heads")
    group = h_q // h_kv
    offs = [int(x) for x in cache_offsets]
    if len(offs) != n_seqs + 1:
        raise OracleArgumentError("one offset per sequence plus one")
    out = np.zeros((n_layers, n_seqs, h_q, values.shape[3]))
    lse = np.zeros((n_layers, n_seqs, h_q))
    for layer in range(n_layers):
        for b in range(n_seqs):
            for h in range(h_q):
                kvh = h // group
                kr = keys[layer, offs[b]:offs[b + 1], kvh]
                vr = values[layer, offs[b]:offs[b + 1], kvh]
                if generated:
                    rows = slice(b * generated, (b + 1) * generated)
                    kr = np.concatenate([kr, np.asarray(k_new, np.float64)[layer, rows, kvh]])
                    vr = np.concatenate([vr, np.asarray(v_new, np.float64)[layer, rows, kvh]])
                out[layer, b, h], lse[layer, b, h] = decode_attention(q[layer, b, h], kr, vr)
    return {"out": out, "lse": lse}
