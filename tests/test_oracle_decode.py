"""Pins for the decode-side oracle (attention of one future query over the
full and the compacted cache, retained mass, position bookkeeping).

Each pin comes from outside the oracle's own formula: the page's printed
example and position table (tests/golden/decode_deletion.json), the exact
decomposition O_full = m O_keep + (1 - m) O_drop and its norm bound, the
invariance under a joint permutation of K and V rows (and the change under a
permutation of V alone), the closed form for equal keys, and consistency with
the selection oracle's own indices and probabilities.
"""

import json
import os

import numpy as np
import pytest

import oracle.decode_oracle as dec
import oracle.snapkv_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "decode_deletion.json")


def _golden():
    return json.load(open(GOLDEN))["printed_on_page"]


def test_page_example_equal_logits():
    """Two equal logits, V = [0, 10]: full output 5, keeping the first gives 0,
    and the kept mass is 1/2."""
    g = _golden()
    keys = np.array([[0.3, -1.2], [0.3, -1.2]])
    values = np.array([[g["equal_logits_values"][0]], [g["equal_logits_values"][1]]], float)
    q = np.array([0.7, 0.4])
    r = dec.decompose(q, keys, values, [0])
    assert r["out_full"][0] == pytest.approx(g["full_output"], abs=1e-12)
    assert r["out_keep"][0] == pytest.approx(g["keep_first_output"], abs=1e-12)
    assert r["m"] == pytest.approx(0.5, abs=1e-15)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_decomposition_identity_and_bound(seed):
    rng = np.random.default_rng(seed)
    n, d = 40, 6
    keys = rng.standard_normal((n, d)) * 1.5
    values = rng.standard_normal((n, d))
    q = rng.standard_normal(d)
    kept = rng.choice(n, size=13, replace=False)
    r = dec.decompose(q, keys, values, kept)
    m = r["m"]
    assert 0.0 < m < 1.0
    np.testing.assert_allclose(r["out_full"], m * r["out_keep"] + (1 - m) * r["out_drop"],
                               rtol=0, atol=1e-13)
    vmax = np.linalg.norm(values, axis=1).max()
    assert r["err"] <= 2 * (1 - m) * vmax + 1e-12
    assert r["err"] == pytest.approx((1 - m) * np.linalg.norm(r["out_drop"] - r["out_keep"]),
                                     abs=1e-13)


def test_mass_from_lse():
    """m equals exp(lse over the kept rows - lse over all rows)."""
    rng = np.random.default_rng(3)
    keys = rng.standard_normal((50, 8)) * 2
    values = rng.standard_normal((50, 8))
    q = rng.standard_normal(8)
    kept = [1, 4, 9, 16, 25, 36, 49]
    _, lse_full = dec.decode_attention(q, keys, values)
    _, lse_keep = dec.decode_attention(q, keys[kept], values[kept])
    assert np.exp(lse_keep - lse_full) == pytest.approx(dec.decompose(q, keys, values, kept)["m"],
                                                         rel=1e-13)


def test_joint_permutation_invariance():
    """Permuting K and V rows together changes nothing; permuting V alone
    changes the output (weights land on the wrong content)."""
    rng = np.random.default_rng(4)
    keys = rng.standard_normal((30, 4))
    values = rng.standard_normal((30, 4))
    q = rng.standard_normal(4) * 2
    perm = rng.permutation(30)
    o1, l1 = dec.decode_attention(q, keys, values)
    o2, l2 = dec.decode_attention(q, keys[perm], values[perm])
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-14)
    assert l2 == pytest.approx(l1, abs=1e-13)
    o3, _ = dec.decode_attention(q, keys, values[perm])
    assert np.abs(o3 - o1).max() > 1e-3


def test_equal_keys_closed_form():
    """All keys equal: uniform weights, output = mean of V, lse = z + log n."""
    rng = np.random.default_rng(5)
    k = rng.standard_normal(5)
    keys = np.tile(k, (17, 1))
    values = rng.standard_normal((17, 3))
    q = rng.standard_normal(5)
    out, lse = dec.decode_attention(q, keys, values)
    np.testing.assert_allclose(out, values.mean(axis=0), rtol=0, atol=1e-14)
    assert lse == pytest.approx(float(k @ q) / np.sqrt(5) + np.log(17), abs=1e-13)


def test_page_position_table():
    g = _golden()
    L, kept = g["prompt_length"], g["kept_positions"]
    c = dec.cache_lengths(L, len(kept), 0)
    assert c["physical_length"] == len(g["physical_slots"])
    assert c["next_logical"] == g["next_logical_position"]
    assert c["next_slot"] == g["next_write_slot"]
    for gen in (1, 7):
        c = dec.cache_lengths(L, len(kept), gen)
        assert c["next_logical"] == L + gen and c["physical_length"] == len(kept) + gen
    # a bypassed prompt (L < C) keeps everything: L + g rows
    assert dec.cache_lengths(3, 5, 2)["physical_length"] == 5


def test_against_the_selection_oracle():
    """Decode over the selection oracle's gathered K/V equals decode over the
    full rows at its indices; the kept mass from the full softmax is at most
    1 and the kept rows' share of the decode weights is exactly 1."""
    rng = np.random.default_rng(6)
    L, W, C, D = 60, 4, 20, 8
    q_win = rng.standard_normal((W, D))
    keys = rng.standard_normal((L, D))
    values = rng.standard_normal((L, D))
    sel = orc.snapkv_head(q_win, keys, values, C, 3, "avg")
    q_future = rng.standard_normal(D)
    o_gathered, l_gathered = dec.decode_attention(q_future, sel["keys"], sel["values"])
    idx = sel["indices"]
    o_idx, l_idx = dec.decode_attention(q_future, keys[idx], values[idx])
    np.testing.assert_allclose(o_gathered, o_idx, rtol=0, atol=1e-14)
    r = dec.decompose(q_future, keys, values, idx)
    assert 0 < r["m"] <= 1
    np.testing.assert_allclose(r["out_keep"], o_idx, rtol=0, atol=1e-13)


def test_packed_layout_and_gqa():
    rng = np.random.default_rng(7)
    layers, S, Hq, Hkv, D, g = 2, 3, 4, 2, 5, 2
    lens = [6, 1, 4]
    offs = np.concatenate([[0], np.cumsum(lens)])
    q = rng.standard_normal((layers, S, Hq, D))
    k = rng.standard_normal((layers, offs[-1], Hkv, D))
    v = rng.standard_normal((layers, offs[-1], Hkv, D))
    kn = rng.standard_normal((layers, S * g, Hkv, D))
    vn = rng.standard_normal((layers, S * g, Hkv, D))
    r = dec.decode_packed(q, k, v, offs, kn, vn, g)
    for layer in range(layers):
        for b in range(S):
            for h in range(Hq):
                kvh = h // 2
                kr = np.concatenate([k[layer, offs[b]:offs[b + 1], kvh], kn[layer, b * g:(b + 1) * g, kvh]])
                vr = np.concatenate([v[layer, offs[b]:offs[b + 1], kvh], vn[layer, b * g:(b + 1) * g, kvh]])
                o, l = dec.decode_attention(q[layer, b, h], kr, vr)
                np.testing.assert_array_equal(r["out"][layer, b, h], o)
                assert r["lse"][layer, b, h] == l


def test_argument_rules():
    with pytest.raises(orc.OracleArgumentError):
        dec.decode_attention(np.zeros(3), np.zeros((0, 3)), np.zeros((0, 3)))
    with pytest.raises(orc.OracleArgumentError):
        dec.decompose(np.zeros(3), np.zeros((4, 3)), np.zeros((4, 3)), [])
    with pytest.raises(orc.OracleArgumentError):
        dec.cache_lengths(4, 0, 0)
