"""Pins for the fp64 oracle: what the SnapKV page and plain mathematics fix.

Each pin comes from outside the oracle: values printed on the page's worked
example and counterexample (tests/golden/*.json, each with its citation),
exact fractions derived by hand from the printed table, harmonic-number closed
forms, probability-mass invariants, and a brute-force checker that takes a
different route (full L x L attention over all queries, subset enumeration).
The mutation tests at the end plant plausible mistakes in the oracle's steps
and check that at least one pin fails for each.
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle.snapkv_oracle as orc
from oracle import bruteforce as bf


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def worked_inputs(g):
    pr = g["printed_on_page"]
    a = [x if x is not None else pr["masked_value_query6_pos7"]
         for x in pr["exp_weights_query6"]]
    b = pr["exp_weights_query7"]
    keys = np.array([[math.log(x), math.log(y)] for x, y in zip(a, b)])
    q_win = np.array([[math.sqrt(2.0), 0.0], [0.0, math.sqrt(2.0)]])
    values = np.array([[float(j), -float(j)] for j in range(len(a))])
    return q_win, keys, values


def counter_inputs(g):
    rc = g["reconstructed"]
    a = [x if x is not None else rc["masked_value_query2_pos3"]
         for x in rc["exp_weights_query2"]]
    b = rc["exp_weights_query3"]
    keys = np.array([[math.log(x), math.log(y)] for x, y in zip(a, b)])
    q_win = np.array([[math.sqrt(2.0), 0.0], [0.0, math.sqrt(2.0)]])
    values = np.arange(len(a) * 2, dtype=np.float64).reshape(len(a), 2)
    return q_win, keys, values


def harmonic(n):
    return sum(Fraction(1, i) for i in range(1, n + 1))


# ---------------------------------------------------------------------------
# Individual pin checks (each returns None or raises AssertionError); the
# mutation tests re-run them against a broken oracle.
# ---------------------------------------------------------------------------

def check_worked_example(g):
    pr, dh = g["printed_on_page"], g["derived_by_hand"]
    q_win, keys, values = worked_inputs(g)
    res = orc.snapkv_head(q_win, keys, values, pr["C"], pr["kernel_size"], pr["pooling"])
    assert res["indices"] == pr["indices"]
    assert np.array_equal(res["values"], values[pr["indices"]])
    assert np.array_equal(res["keys"], keys[pr["indices"]])
    np.testing.assert_allclose(orc.window_row_exp_sums(q_win, keys), pr["row_sums"], rtol=1e-12)
    exp_votes = [float(Fraction(x)) for x in dh["votes"]]
    exp_pooled = [float(Fraction(x)) for x in dh["pooled_avg3"]]
    np.testing.assert_allclose(res["votes"], exp_votes, rtol=1e-12, atol=0)
    np.testing.assert_allclose(res["pooled"], exp_pooled, rtol=1e-12, atol=0)
    assert int(np.argmax(res["votes"])) == pr["raw_vote_top"]
    assert int(np.argmax(res["pooled"])) == pr["pooled_top"]
    mx = orc.snapkv_head(q_win, keys, values, pr["C"], 3, "max")
    np.testing.assert_allclose(mx["pooled"], [float(Fraction(x)) for x in dh["pooled_max3"]],
                               rtol=1e-12, atol=0)
    assert mx["indices"] == dh["indices_max3"]


def check_counterexample(g):
    pr, rc = g["printed_on_page"], g["reconstructed"]
    q_win, keys, values = counter_inputs(g)
    res = orc.snapkv_head(q_win, keys, values, rc["C"], rc["kernel_size"], rc["pooling"])
    np.testing.assert_allclose(res["votes"], [pr["vote_A"], pr["vote_B"]], rtol=1e-12)
    np.testing.assert_allclose(res["probs"][0, :2], pr["vote_A_terms"][:1] + pr["vote_B_terms"][:1],
                               rtol=1e-12)
    np.testing.assert_allclose(res["probs"][1, :2], pr["vote_A_terms"][1:] + pr["vote_B_terms"][1:],
                               rtol=1e-12)
    assert res["indices"] == rc["indices"]          # B (position 1) kept
    # The other algorithm the page warns about, computed from the table by plain
    # arithmetic: normalising each row over the prefix columns only keeps A.
    rows = [[9, 1], [9, 27]]
    alt = [sum(Fraction(r[j], sum(r)) for r in rows) for j in range(2)]
    assert [float(x) for x in alt] == pytest.approx([pr["prefix_only_A"], pr["prefix_only_B"]])
    assert alt[0] > alt[1] and res["votes"][1] > res["votes"][0]


def check_uniform_closed_form(length=40, window=5, capacity=13, kernel=5, dim=3):
    """All keys equal => row r sees P+r+1 equal logits => s_j = H_L - H_P."""
    rng = np.random.default_rng(7)
    q_win = rng.standard_normal((window, dim))
    keys = np.tile(rng.standard_normal(dim), (length, 1))
    values = rng.standard_normal((length, dim))
    res = orc.snapkv_head(q_win, keys, values, capacity, kernel, "avg")
    prefix, radius = length - window, kernel // 2
    s = float(harmonic(length) - harmonic(prefix))
    np.testing.assert_allclose(res["votes"], np.full(prefix, s), rtol=1e-13)
    expect = [s * (min(j, radius) + 1 + min(prefix - 1 - j, radius)) / kernel
              for j in range(prefix)]
    np.testing.assert_allclose(res["pooled"], expect, rtol=1e-13)
    # interior scores tie exactly in exact arithmetic; fp64 sums of equal terms
    # in a fixed order tie bit for bit, so the smallest-index rule decides.
    n_keep = capacity - window
    assert res["indices"] == list(range(radius, radius + n_keep)) + list(range(prefix, length))


def check_edge_divisor(kernel=7):
    """pooled[0] = (s_0 + ... + s_R) / k: out-of-range cells add zero, divisor stays k."""
    rng = np.random.default_rng(11)
    s = rng.random(20)
    pooled = orc.pool_scores(s, kernel, "avg")
    r = kernel // 2
    assert pooled[0] == pytest.approx(sum(s[: r + 1]) / kernel, rel=1e-14)
    assert pooled[-1] == pytest.approx(sum(s[-(r + 1):]) / kernel, rel=1e-14)
    assert pooled[r] == pytest.approx(sum(s[: 2 * r + 1]) / kernel, rel=1e-14)
    assert orc.pool_scores(s, 1, "avg").tolist() == s.tolist()


def run_all_pins(golden_dir):
    check_worked_example(_load(golden_dir, "worked_example.json"))
    check_counterexample(_load(golden_dir, "counterexample.json"))
    check_uniform_closed_form()
    check_edge_divisor()
    check_bruteforce_cases()


# ---------------------------------------------------------------------------
# Tests
# ---------------------------------------------------------------------------

def test_worked_example(golden_dir):
    check_worked_example(_load(golden_dir, "worked_example.json"))


def test_counterexample(golden_dir):
    check_counterexample(_load(golden_dir, "counterexample.json"))


def test_counterexample_pooled_tie_needs_width_one(golden_dir):
    """With avg width 3 the two prefix scores tie at exactly 1/3 and A wins the tie."""
    g = _load(golden_dir, "counterexample.json")
    q_win, keys, values = counter_inputs(g)
    res = orc.snapkv_head(q_win, keys, values, 3, 3, "avg")
    np.testing.assert_allclose(res["pooled"], [1.0 / 3, 1.0 / 3], rtol=1e-14)
    assert res["indices"] == [0, 2, 3]


def test_uniform_closed_form():
    check_uniform_closed_form()
    check_uniform_closed_form(length=64, window=16, capacity=20, kernel=3, dim=8)


def test_zero_queries_same_as_uniform():
    """q_win = 0 gives all-zero logits: the same harmonic closed form."""
    rng = np.random.default_rng(3)
    length, window = 30, 4
    res = orc.snapkv_head(np.zeros((window, 6)), rng.standard_normal((length, 6)),
                          rng.standard_normal((length, 6)), 10, 1, "avg")
    s = float(harmonic(length) - harmonic(length - window))
    np.testing.assert_allclose(res["votes"], s, rtol=1e-13)


def test_edge_divisor():
    check_edge_divisor()
    check_edge_divisor(3)


def test_pool_wider_than_prefix():
    """k > P: every neighbour is in range for every j; divisor is still k."""
    s = np.array([0.5, 0.25, 0.125])
    np.testing.assert_allclose(orc.pool_scores(s, 9, "avg"), [0.875 / 9] * 3, rtol=1e-15)
    assert orc.pool_scores(s, 9, "max").tolist() == [0.5] * 3


def test_probability_mass_invariants():
    rng = np.random.default_rng(5)
    for length, window in [(50, 7), (33, 1), (9, 9 - 1)]:
        q_win = rng.standard_normal((window, 4)) * 2
        keys = rng.standard_normal((length, 4)) * 2
        res = orc.snapkv_head(q_win, keys, keys, length, 3, "avg")
        p = res["probs"]
        prefix = length - window
        for r in range(window):
            assert p[r, : prefix + r + 1].sum() == pytest.approx(1.0, abs=1e-13)
            assert np.all(p[r, prefix + r + 1:] == 0)
        window_mass = sum(p[r, prefix:prefix + r + 1].sum() for r in range(window))
        assert res["votes"].sum() == pytest.approx(window - window_mass, abs=1e-12)
        assert res["votes"].sum() <= window + 1e-12
        assert np.all(res["votes"] >= 0)


def test_bypass_and_equal_capacity():
    rng = np.random.default_rng(9)
    q_win, keys, values = (rng.standard_normal((3, 4)), rng.standard_normal((10, 4)),
                           rng.standard_normal((10, 4)))
    res = orc.snapkv_head(q_win, keys, values, 11, 3, "avg")     # L < C
    assert res["indices"] == list(range(10))
    assert np.array_equal(res["values"], values) and np.array_equal(res["keys"], keys)
    res = orc.snapkv_head(q_win, keys, values, 10, 3, "avg")     # L == C: normal path
    assert sorted(res["indices"]) == list(range(10))
    assert res["indices"][-3:] == [7, 8, 9]
    order = res["indices"][:7]
    assert order == sorted(range(7), key=lambda j: (-res["pooled"][j], j))


def check_bruteforce_cases(n_cases=12):
    rng = np.random.default_rng(2024)
    done = 0
    while done < n_cases:
        length = int(rng.integers(4, 13))
        window = int(rng.integers(1, length))
        capacity = int(rng.integers(window + 1, length + 1))
        kernel = int(rng.choice([1, 3, 5]))
        pooling = str(rng.choice(["avg", "max"]))
        dim = int(rng.integers(1, 5))
        queries = rng.standard_normal((length, dim)) * 1.5
        keys = rng.standard_normal((length, dim)) * 1.5
        values = rng.standard_normal((length, dim))
        res = orc.snapkv_head(queries[length - window:], keys, values, capacity, kernel, pooling)
        brute = bf.snapkv_bruteforce(queries.tolist(), keys.tolist(), window, capacity,
                                     kernel, pooling)
        np.testing.assert_allclose(res["votes"], brute["votes"], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(res["pooled"], brute["pooled"], rtol=1e-12, atol=1e-15)
        sp = sorted(brute["pooled"], reverse=True)
        n_keep = capacity - window
        if n_keep < len(sp) and sp[n_keep - 1] - sp[n_keep] < 1e-9:
            continue                      # near tie: fp64 route differences may flip it
        assert res["indices"] == brute["indices"]
        att = np.array(brute["attention"])
        np.testing.assert_allclose(res["probs"], att[length - window:], rtol=1e-12, atol=1e-15)
        done += 1


def test_bruteforce_agreement():
    check_bruteforce_cases()


def test_bruteforce_exact_ties():
    """Duplicated keys give exact ties; both routes keep the smaller index."""
    length, window, capacity = 10, 2, 5
    keys = np.array([[0.3, 0.1]] * 4 + [[1.0, -0.5]] * 4 + [[0.2, 0.2], [0.0, 1.0]])
    queries = np.tile([[0.7, -0.2]], (length, 1))
    res = orc.snapkv_head(queries[-window:], keys, keys, capacity, 1, "avg")
    brute = bf.snapkv_bruteforce(queries.tolist(), keys.tolist(), window, capacity, 1, "avg")
    assert res["indices"] == brute["indices"] == [4, 5, 6, 8, 9]


def test_per_head_independence_and_pairing():
    """Two heads with different key layouts keep different positions; K and V
    are gathered with the same indices (V row j encodes j)."""
    length, window, capacity, dim = 24, 4, 10, 4
    q = np.zeros((1, window, 2, dim))
    q[0, :, :, 0] = 3.0
    keys = np.zeros((1, length, 2, dim))
    keys[0, 2:6, 0, 0] = 1.0                 # head 0 looks at the front
    keys[0, 12:16, 1, 0] = 1.0               # head 1 looks at the middle
    values = np.zeros((1, length, 2, dim))
    values[0, :, :, 0] = np.arange(length)[:, None]
    values[0, :, :, 1] = np.arange(2)[None, :]
    out = orc.snapkv_packed(q, keys, values, [0, length], window, capacity, 1, "avg")
    idx = out["out_idx"][0]
    assert set(idx[:4, 0]) == {2, 3, 4, 5}
    assert set(idx[:4, 1]) == {12, 13, 14, 15}
    assert np.array_equal(out["out_V"][0, :, :, 0], idx.astype(np.float64))
    assert np.array_equal(out["out_V"][0, :, :, 1], np.tile([0.0, 1.0], (capacity, 1)))
    assert np.array_equal(out["out_K"][0, :, 0], keys[0, idx[:, 0], 0])


def test_packed_ragged_matches_single_heads():
    rng = np.random.default_rng(17)
    lens, window, capacity, heads, dim, layers = [9, 3, 14], 3, 8, 2, 3, 2
    offs = np.concatenate([[0], np.cumsum(lens)])
    q = rng.standard_normal((layers, len(lens) * window, heads, dim))
    keys = rng.standard_normal((layers, offs[-1], heads, dim))
    values = rng.standard_normal((layers, offs[-1], heads, dim))
    out = orc.snapkv_packed(q, keys, values, offs, window, capacity, 3, "max")
    assert out["out_idx"].shape == (layers, 8 + 3 + 8, heads)
    for layer in range(layers):
        for b, length in enumerate(lens):
            for h in range(heads):
                r = orc.snapkv_head(q[layer, b * window:(b + 1) * window, h],
                                    keys[layer, offs[b]:offs[b + 1], h],
                                    values[layer, offs[b]:offs[b + 1], h], capacity, 3, "max")
                oo = out["out_offsets"][b]
                n = len(r["indices"])
                assert out["out_idx"][layer, oo:oo + n, h].tolist() == r["indices"]
    assert out["out_idx"][0, 8:11, 0].tolist() == [0, 1, 2]      # L=3 < C: bypass


def test_select_from_pooled_ties_and_bypass():
    pooled = np.array([0.5, 0.25, 0.5, 0.75, 0.25, 0.5], dtype=np.float32).astype(np.float64)
    assert orc.select_from_pooled(pooled, 8, 2, 5) == [3, 0, 2, 6, 7]
    assert orc.select_from_pooled(pooled, 8, 2, 9) == list(range(8))
    assert orc.select_from_pooled(pooled, 8, 2, 8) == [3, 0, 2, 5, 1, 4, 6, 7]


@pytest.mark.parametrize("bad", [
    dict(length=0), dict(vlen=5), dict(dim=0), dict(nonfinite="k"), dict(nonfinite="v"),
    dict(nonfinite="q"), dict(window=7), dict(capacity=3), dict(kernel=2), dict(kernel=0),
    dict(pooling="sum"), dict(capacity=4.0),
])
def test_argument_rules(bad):
    length = bad.get("length", 6)
    dim = bad.get("dim", 2)
    window = bad.get("window", 3)
    q = np.ones((min(window, 7), dim))
    k = np.ones((length, dim))
    v = np.ones((bad.get("vlen", length), dim))
    if bad.get("nonfinite") == "k":
        k[1, 0] = np.inf
    if bad.get("nonfinite") == "v":
        v[1, 0] = np.nan
    if bad.get("nonfinite") == "q":
        q[0, 0] = np.nan
    with pytest.raises(orc.OracleArgumentError):
        orc.snapkv_head(q, k, v, bad.get("capacity", 5), bad.get("kernel", 3),
                        bad.get("pooling", "avg"))


def test_nonfinite_dot_product_is_an_error():
    big = np.array([[1e200, 1e200]])
    with pytest.raises(orc.OracleArgumentError):
        orc.snapkv_head(big, np.ones((4, 2)) * 1e200, np.ones((4, 2)), 3, 1, "avg")


def test_window_equal_to_prompt_is_valid_when_bypassed():
    res = orc.snapkv_head(np.ones((4, 2)), np.ones((4, 2)), np.ones((4, 2)), 5, 1, "avg")
    assert res["indices"] == [0, 1, 2, 3]


# ---------------------------------------------------------------------------
# Planted mistakes: each plausible bug must make some pin fail.
# ---------------------------------------------------------------------------

def _no_causal_mask(z):
    e = np.exp(z - z.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def _prefix_only_normalisation(z):
    w, l = z.shape
    p = np.zeros_like(z)
    for r in range(w):
        pre = z[r, : l - w]
        e = np.exp(pre - pre.max())
        p[r, : l - w] = e / e.sum()
    return p


def _row_is_position_r(z):
    w, l = z.shape
    p = np.zeros_like(z)
    for r in range(w):
        vis = z[r, : r + 1]
        e = np.exp(vis - vis.max())
        p[r, : r + 1] = e / e.sum()
    return p


def _avg_by_inrange_count(original):
    def pool(s, k, pooling):
        if pooling != "avg":
            return original(s, k, pooling)
        r = k // 2
        return np.array([s[max(0, j - r): j + r + 1].mean() for j in range(len(s))])
    return pool


def _unscaled_logits(q_win, keys):
    return q_win @ keys.T


def _largest_index_first(pooled, n):
    return sorted(range(len(pooled)), key=lambda j: (-pooled[j], -j))[:n]


def _mean_votes(p):
    w, l = p.shape
    return p[:, : l - w].mean(axis=0)


def _plain(fn):
    return lambda original: fn


MUTATIONS = {
    "no_causal_mask": ("causal_probabilities", _plain(_no_causal_mask)),
    "prefix_only_softmax": ("causal_probabilities", _plain(_prefix_only_normalisation)),
    "row_r_is_position_r": ("causal_probabilities", _plain(_row_is_position_r)),
    "avg_divides_by_inrange": ("pool_scores", _avg_by_inrange_count),
    "missing_inv_sqrt_d": ("window_logits", _plain(_unscaled_logits)),
    "ties_to_larger_index": ("top_prefix", _plain(_largest_index_first)),
    "votes_averaged": ("prefix_votes", _plain(_mean_votes)),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, golden_dir, monkeypatch):
    attr, factory = MUTATIONS[name]
    monkeypatch.setattr(orc, attr, factory(getattr(orc, attr)))
    with pytest.raises(AssertionError):
        run_all_pins(golden_dir)


def test_all_pins_pass_unmutated(golden_dir):
    run_all_pins(golden_dir)
