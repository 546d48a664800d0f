"""Pins for the reverse-mask attention oracle (counter-causal scorer).

Each pin comes from outside the oracle's own loop: the decode oracle (pinned
on its own page example) over each query's future rows; PyTorch's scaled
dot-product attention with an explicit strictly-upper mask; the closed form
for equal keys (the mean of the later values, log of their count); the
boundary rows (the last position has no future, the second to last sees
only the last); a joint permutation of rows and positions; dependence on
later rows only; and planted mistakes that one of these catches.
"""

import numpy as np
import pytest
import torch

import oracle.decode_oracle as dec
import oracle.reverse_oracle as rev
from oracle.snapkv_oracle import OracleArgumentError


def _head(n, d, seed, dv=None):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((n, d)), rng.standard_normal((n, d)),
            rng.standard_normal((n, dv or d)))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_decode_oracle_on_the_future_rows(seed):
    q, k, v = _head(23, 8, seed)
    out, lse = rev.reverse_attention(q, k, v)
    for i in range(22):
        o, l = dec.decode_attention(q[i], k[i + 1:], v[i + 1:])
        np.testing.assert_allclose(out[i], o, rtol=1e-12, atol=1e-13)
        assert lse[i] == pytest.approx(l, rel=1e-12)


def test_matches_library_attention_with_an_upper_mask():
    q, k, v = _head(40, 16, 7, dv=5)
    out, lse = rev.reverse_attention(q, k, v)
    mask = torch.ones(40, 40, dtype=torch.bool).triu(1)          # row i: columns j > i
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q)[None], torch.tensor(k)[None], torch.tensor(v)[None], attn_mask=mask[None])
    np.testing.assert_allclose(out[:-1], ref[0, :-1].numpy(), rtol=1e-10, atol=1e-12)
    s = torch.tensor(q) @ torch.tensor(k).T / 4.0
    ref_lse = torch.logsumexp(s.masked_fill(~mask, float("-inf")), dim=1)
    np.testing.assert_allclose(lse[:-1], ref_lse[:-1].numpy(), rtol=1e-12)


def test_equal_keys_closed_form():
    """All keys equal: every later row gets the same weight, so out_i is the
    mean of v_{i+1..n-1} and lse_i = q_i . k / sqrt(D) + log(n - 1 - i)."""
    n, d = 17, 4
    rng = np.random.default_rng(3)
    k = np.tile(rng.standard_normal(d), (n, 1))
    q = rng.standard_normal((n, d))
    v = rng.standard_normal((n, 3))
    out, lse = rev.reverse_attention(q, k, v)
    for i in range(n - 1):
        np.testing.assert_allclose(out[i], v[i + 1:].mean(axis=0), rtol=1e-12, atol=1e-14)
        assert lse[i] == pytest.approx(q[i] @ k[0] / 2.0 + np.log(n - 1 - i), rel=1e-12)


def test_boundary_rows():
    q, k, v = _head(6, 4, 4)
    out, lse = rev.reverse_attention(q, k, v)
    assert np.all(out[-1] == 0) and lse[-1] == -np.inf          # no future: largest surprise
    np.testing.assert_allclose(out[-2], v[-1], rtol=1e-15)     # one later row: weight 1
    assert lse[-2] == pytest.approx(q[-2] @ k[-1] / 2.0, rel=1e-14)
    o1, l1 = rev.reverse_attention(q[:1], k[:1], v[:1])         # a one-row sequence
    assert np.all(o1 == 0) and l1[0] == -np.inf


def test_positions_follow_rows_through_a_permutation():
    """Algorithm 3 reorders the memory by surprise: the mask follows the
    original positions, so permuting rows and positions together permutes the
    outputs."""
    q, k, v = _head(19, 8, 5)
    out, lse = rev.reverse_attention(q, k, v)
    perm = np.random.default_rng(6).permutation(19)
    out_p, lse_p = rev.reverse_attention(q[perm], k[perm], v[perm], positions=perm)
    np.testing.assert_allclose(out_p, out[perm], rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(np.isinf(lse_p), np.isinf(lse[perm]))
    fin = np.isfinite(lse_p)
    np.testing.assert_allclose(lse_p[fin], lse[perm][fin], rtol=1e-12)
    # gaps in the positions change nothing (only their order matters)
    out_g, _ = rev.reverse_attention(q, k, v, positions=np.arange(19) * 7 + 100)
    np.testing.assert_allclose(out_g, out, rtol=0, atol=0)


def test_depends_on_later_rows_only():
    q, k, v = _head(12, 4, 8)
    out, _ = rev.reverse_attention(q, k, v)
    k2, v2 = k.copy(), v.copy()
    k2[:5] += 3.0
    v2[:5] -= 2.0
    out2, _ = rev.reverse_attention(q, k2, v2)
    np.testing.assert_allclose(out2[4:], out[4:], rtol=0, atol=0)   # rows >= 4 see only j >= 5
    assert np.abs(out2[:4] - out[:4]).max() > 1e-3


def test_packed_layers_heads_and_groups():
    rng = np.random.default_rng(9)
    L, T, H, Hkv, D = 2, 30, 4, 2, 8
    q = rng.standard_normal((L, T, H, D))
    k = rng.standard_normal((L, T, Hkv, D))
    v = rng.standard_normal((L, T, Hkv, D))
    offs = [0, 11, 11, 30]
    r = rev.reverse_packed(q, k, v, offs)
    for layer in range(L):
        for b in range(3):
            a, e = offs[b], offs[b + 1]
            for h in range(H):
                o, l = rev.reverse_attention(q[layer, a:e, h], k[layer, a:e, h // 2],
                                             v[layer, a:e, h // 2]) if e > a else (None, None)
                if e > a:
                    np.testing.assert_array_equal(r["out"][layer, a:e, h], o)
                    np.testing.assert_array_equal(r["lse"][layer, h, a:e], l)
    with pytest.raises(OracleArgumentError):
        rev.reverse_packed(q, k[:, :, :1].repeat(3, axis=2), v[:, :, :1].repeat(3, axis=2), offs)
    with pytest.raises(OracleArgumentError):
        rev.reverse_attention(q[0, :, 0], k[0, :, 0], v[0, :, 0], positions=[0] * T)


def test_planted_mistakes_fail_a_pin():
    """Three plausible bugs: the diagonal included (j >= i), the causal
    direction (j < i), the scale left out. Each breaks the boundary or
    closed-form pins."""
    n, d = 9, 4
    rng = np.random.default_rng(10)
    k = np.tile(rng.standard_normal(d), (n, 1))
    q, v = rng.standard_normal((n, d)), rng.standard_normal((n, 2))

    def variant(keep, scale):
        out = np.zeros((n, 2))
        lse = np.full(n, -np.inf)
        for i in range(n):
            sel = keep(np.arange(n), i)
            if sel.any():
                z = k[sel] @ q[i] * scale
                out[i] = (np.exp(z - z.max()) / np.exp(z - z.max()).sum()) @ v[sel]
                lse[i] = z.max() + np.log(np.exp(z - z.max()).sum())
        return out, lse

    def pins_hold(out, lse):
        ok = np.all(out[-1] == 0) and lse[-1] == -np.inf
        for i in range(n - 1):
            ok &= np.allclose(out[i], v[i + 1:].mean(axis=0), atol=1e-12)
            ok &= np.isclose(lse[i], q[i] @ k[0] / 2.0 + np.log(n - 1 - i), rtol=1e-12)
        return bool(ok)

    assert pins_hold(*rev.reverse_attention(q, k, v))
    assert not pins_hold(*variant(lambda j, i: j >= i, 0.5))
    assert not pins_hold(*variant(lambda j, i: j < i, 0.5))
    assert not pins_hold(*variant(lambda j, i: j > i, 1.0))


def test_outputs_are_convex_combinations_of_later_values():
    q, k, v = _head(31, 8, 12, dv=4)
    out, _ = rev.reverse_attention(q * 3.0, k, v)
    for i in range(30):
        lo, hi = v[i + 1:].min(axis=0), v[i + 1:].max(axis=0)
        assert np.all(out[i] >= lo - 1e-12) and np.all(out[i] <= hi + 1e-12)
