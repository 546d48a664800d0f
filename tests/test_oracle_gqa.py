"""Pins for the grouped-query (GQA) oracle.

The page's section on GQA ("GQA 下的缓存节省不能只算 C 除以 L") fixes the
expanded (repeat_kv) integration: select per query head on K/V expanded to the
query heads. The group-shared selection is our reading (votes of the G query
heads summed, then pooled and selected once). Each pin comes from outside the
group code: the expansion identity, the reduction to one head at G = 1, the
exact doubling of votes for two identical heads, the harmonic-number closed
form with all keys equal, and the brute-force route (full L x L attention of
every query head, summed, explicitly padded pooling, subset enumeration).
"""

from fractions import Fraction

import numpy as np
import pytest

import oracle.snapkv_oracle as orc
import oracle.gqa_oracle as gq
from oracle import bruteforce as bf


def _rand_packed(seed, lens, window, h_q, h_kv, dim, layers):
    rng = np.random.default_rng(seed)
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(int)
    q = rng.standard_normal((layers, len(lens) * window, h_q, dim))
    k = rng.standard_normal((layers, offs[-1], h_kv, dim))
    v = rng.standard_normal((layers, offs[-1], h_kv, dim))
    return q, k, v, offs


def test_repeat_mode_equals_expanded_cache():
    """repeat: identical to the per-head oracle on K/V expanded with repeat_kv."""
    q, k, v, offs = _rand_packed(3, [12, 5, 20], 3, 4, 2, 4, 2)
    out = gq.snapkv_packed_gqa(q, k, v, offs, 3, 9, 3, "avg", "repeat")
    ke, ve = np.repeat(k, 2, axis=2), np.repeat(v, 2, axis=2)
    ref = orc.snapkv_packed(q, ke, ve, offs, 3, 9, 3, "avg")
    for name in ("out_idx", "out_K", "out_V", "votes", "pooled"):
        np.testing.assert_array_equal(out[name], ref[name])


def test_group_of_one_is_the_single_head():
    rng = np.random.default_rng(4)
    qg = rng.standard_normal((1, 3, 5))
    keys = rng.standard_normal((30, 5))
    vals = rng.standard_normal((30, 5))
    g = gq.snapkv_group(qg, keys, vals, 12, 5, "max")
    h = orc.snapkv_head(qg[0], keys, vals, 12, 5, "max")
    assert g["indices"] == h["indices"]
    np.testing.assert_array_equal(g["votes"], h["votes"])
    np.testing.assert_array_equal(g["pooled"], h["pooled"])


@pytest.mark.parametrize("pooling", ["avg", "max"])
def test_two_identical_heads_double_the_votes(pooling):
    """Two equal query heads: summed votes are exactly twice one head's (doubling
    is exact in binary floating point), so pooled scores double and the
    selection is unchanged."""
    rng = np.random.default_rng(5)
    q1 = rng.standard_normal((4, 6))
    keys = rng.standard_normal((40, 6))
    vals = rng.standard_normal((40, 6))
    g = gq.snapkv_group(np.stack([q1, q1]), keys, vals, 15, 3, pooling)
    h = orc.snapkv_head(q1, keys, vals, 15, 3, pooling)
    np.testing.assert_array_equal(g["votes"], 2.0 * h["votes"])
    np.testing.assert_array_equal(g["pooled"], 2.0 * h["pooled"])
    assert g["indices"] == h["indices"]


def test_group_uniform_closed_form():
    """All keys equal: each visible column of row r has probability 1/(P+r+1),
    so each head votes H_L - H_P for every prefix j and the group G times that;
    interior avg-pooled scores tie exactly and the smallest positions from R win."""
    length, window, capacity, kernel, group = 40, 4, 14, 5, 3
    rng = np.random.default_rng(6)
    qg = rng.standard_normal((group, window, 3))
    keys = np.tile(rng.standard_normal((1, 3)), (length, 1))
    g = gq.snapkv_group(qg, keys, keys, capacity, kernel, "avg")
    prefix = length - window
    s = sum(Fraction(1, i) for i in range(prefix + 1, length + 1))
    np.testing.assert_allclose(g["votes"], group * float(s), rtol=1e-13)
    r = kernel // 2
    assert g["indices"][:capacity - window] == list(range(r, r + capacity - window))
    assert g["indices"][capacity - window:] == list(range(prefix, length))


def test_group_brute_force():
    """Tiny groups against the brute-force route (full attention of every query
    head, summed per column, padded pooling, subset enumeration)."""
    rng = np.random.default_rng(7)
    cases = [(9, 2, 5, 3, 2, 2, "avg"), (11, 3, 6, 1, 3, 3, "max"), (10, 2, 7, 3, 2, 4, "avg")]
    for length, window, capacity, kernel, dim, group, pooling in cases:
        queries = rng.standard_normal((group, length, dim))
        keys = rng.standard_normal((length, dim))
        g = gq.snapkv_group(queries[:, length - window:], keys, keys, capacity, kernel, pooling)
        votes = None
        for h in range(group):
            att = bf.full_causal_attention(queries[h].tolist(), keys.tolist())
            vh = bf.votes_from_attention(att, window)
            votes = vh if votes is None else [a + b for a, b in zip(votes, vh)]
        pooled = bf.pool_padded(votes, kernel, pooling)
        kept = bf.kept_prefix_by_enumeration(pooled, capacity - window)
        assert g["indices"] == kept + list(range(length - window, length))
        np.testing.assert_allclose(g["votes"], votes, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(g["pooled"], pooled, rtol=1e-12, atol=1e-15)


def test_group_decides_on_the_sum():
    """Head 0 prefers position 2, head 1 position 9; with one prefix slot the
    group keeps whichever has the larger summed vote, which can be neither
    head's own choice."""
    length, window, capacity, dim = 16, 2, 3, 4
    keys = np.zeros((length, dim))
    keys[2, 0] = 1.0
    keys[9, 1] = 1.0
    keys[5, 0] = keys[5, 1] = 0.8       # liked a little by both heads
    q = np.zeros((2, window, dim))
    q[0, :, 0] = 4.0
    q[1, :, 1] = 4.0
    g = gq.snapkv_group(q, keys, keys, capacity, 1, "avg")
    h0 = orc.snapkv_head(q[0], keys, keys, capacity, 1, "avg")
    h1 = orc.snapkv_head(q[1], keys, keys, capacity, 1, "avg")
    assert h0["indices"][0] == 2 and h1["indices"][0] == 9
    summed = h0["votes"] + h1["votes"]
    assert g["indices"][0] == int(np.argmax(summed))


def test_group_bypass_and_argument_rules():
    rng = np.random.default_rng(8)
    q = rng.standard_normal((2, 3, 4))
    keys = rng.standard_normal((5, 4))
    g = gq.snapkv_group(q, keys, keys, 8, 3, "avg")
    assert g["indices"] == [0, 1, 2, 3, 4]
    with pytest.raises(orc.OracleArgumentError):
        gq.snapkv_group(q, keys, keys, 8, 2, "avg")            # even width
    with pytest.raises(orc.OracleArgumentError):
        gq.snapkv_packed_gqa(np.zeros((1, 3, 3, 4)), np.zeros((1, 5, 2, 4)),
                             np.zeros((1, 5, 2, 4)), [0, 5], 3, 4, 1, "avg", "group")


def test_packed_group_layout():
    q, k, v, offs = _rand_packed(9, [10, 4, 13], 2, 6, 2, 3, 2)
    out = gq.snapkv_packed_gqa(q, k, v, offs, 2, 6, 3, "avg", "group")
    assert out["out_idx"].shape == (2, 6 + 4 + 6, 2)
    for layer in range(2):
        for b, length in enumerate([10, 4, 13]):
            for h in range(2):
                qg = np.stack([q[layer, b * 2:(b + 1) * 2, h * 3 + j] for j in range(3)])
                r = gq.snapkv_group(qg, k[layer, offs[b]:offs[b + 1], h],
                                    v[layer, offs[b]:offs[b + 1], h], 6, 3, "avg")
                oo = out["out_offsets"][b]
                n = len(r["indices"])
                assert out["out_idx"][layer, oo:oo + n, h].tolist() == r["indices"]
                np.testing.assert_array_equal(out["out_V"][layer, oo:oo + n, h], r["values"])
