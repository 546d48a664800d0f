"""Brute-force checker for tiny SnapKV inputs (pure Python loops, fp64).

TEST INFRASTRUCTURE, like the rest of ``oracle/``. It shares nothing with
``snapkv_oracle`` and follows a different route to the same quantities:

* it builds the full L x L causal attention matrix from ALL L queries (the
  attention every prompt position would compute) and only then keeps the last
  W rows, instead of scoring the window rows alone;
* it pools with an explicitly zero-padded copy of the vote array;
* it finds the kept prefix set by enumerating every (C - W)-subset and keeping
  the one subset whose members all precede every non-member in the
  (-score, index) order, instead of sorting.

Source: page "SnapKV: choosing the KV cache of a long prompt with an
observation window", sections "Votes must come from the full-prompt causal
softmax" (投票必须来自完整提示词的因果 softmax) and "Pooling turns a peak into a
neighbourhood preference" (池化把一个峰值扩展成邻域偏好).
Use only for L up to a few dozen and C(P, C-W) up to about 1e5.
"""

from __future__ import annotations

import itertools
import math
from typing import List, Sequence


def full_causal_attention(queries: Sequence[Sequence[float]],
                          keys: Sequence[Sequence[float]]) -> List[List[float]]:
    """A[t][j] = softmax over j <= t of q_t . k_j / sqrt(D); A[t][j] = 0 for j > t."""
    length = len(keys)
    dim = len(keys[0])
    scale = 1.0 / math.sqrt(dim)
    att = [[0.0] * length for _ in range(length)]
    for t in range(length):
        logits = [math.fsum(queries[t][d] * keys[j][d] for d in range(dim)) * scale
                  for j in range(t + 1)]
        top = max(logits)
        weights = [math.exp(x - top) for x in logits]
        total = math.fsum(weights)
        for j in range(t + 1):
            att[t][j] = weights[j] / total
    return att


def votes_from_attention(att: List[List[float]], window: int) -> List[float]:
    """Sum of the last W rows of the attention matrix over each prefix column."""
    length = len(att)
    prefix = length - window
    return [math.fsum(att[t][j] for t in range(prefix, length)) for j in range(prefix)]


def pool_padded(votes: List[float], kernel_size: int, pooling: str) -> List[float]:
    """Slide a width-k window over [0]*R + votes + [0]*R (avg divides by k).

    For max, padding cells are skipped, which equals zero padding since votes
    are non-negative.
    """
    radius = kernel_size // 2
    padded = [None] * radius + list(votes) + [None] * radius
    out = []
    for j in range(len(votes)):
        cells = padded[j: j + kernel_size]
        if pooling == "avg":
            out.append(math.fsum(c for c in cells if c is not None) / kernel_size)
        else:
            out.append(max(c for c in cells if c is not None))
    return out


def kept_prefix_by_enumeration(pooled: List[float], n_keep: int) -> List[int]:
    """The unique n_keep-subset S with key(i) < key(o) for all i in S, o not in S.

    key(j) = (-pooled[j], j). Returns S in key order.
    """
    prefix = len(pooled)

    def key(j):
        return (-pooled[j], j)

    found = []
    for subset in itertools.combinations(range(prefix), n_keep):
        inside = set(subset)
        worst_in = max(key(j) for j in subset)
        if all(worst_in < key(o) for o in range(prefix) if o not in inside):
            found.append(subset)
    assert len(found) == 1, f"expected exactly one dominant subset, got {len(found)}"
    return sorted(found[0], key=key)


def snapkv_bruteforce(queries, keys, window: int, capacity: int,
                      kernel_size: int, pooling: str):
    """Indices, votes and pooled scores for one head from the full attention."""
    length = len(keys)
    if length < capacity:
        return {"indices": list(range(length)), "votes": [], "pooled": []}
    att = full_causal_attention(queries, keys)
    votes = votes_from_attention(att, window)
    pooled = pool_padded(votes, kernel_size, pooling)
    prefix = length - window
    kept = kept_prefix_by_enumeration(pooled, capacity - window)
    return {"indices": kept + list(range(prefix, length)), "votes": votes,
            "pooled": pooled, "attention": att}
