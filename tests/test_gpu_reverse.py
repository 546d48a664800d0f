"""Reverse-mask attention (counter-causal scorer) on the GPU against the fp64
oracle.

Bars: out within 1e-4 relative plus 2e-5 absolute, lse within 1e-4 absolute
(fp32 logits and sums over the same bf16 inputs the oracle reads in fp64; P
applied as a bf16 hi + lo pair, so its rounding stays near 2^-17 of each
weight); rows with no later position exactly out = 0 and lse = -inf.
"""

import numpy as np
import pytest
import torch

import oracle
from helpers import ensure_built

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def api():
    from kv_cache_eviction_snapkv_gb300 import api as a
    return a


def assert_ok():
    st = api().kvsel_device_status()
    assert st == 0, api().kvsel_status_string(st)


def f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def inputs(layers, T, H, Hkv, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn((layers, T, H, 128), generator=g) * scale).to(torch.bfloat16)
    k = (torch.randn((layers, T, Hkv, 128), generator=g) * scale).to(torch.bfloat16)
    v = torch.randn((layers, T, Hkv, 128), generator=g).to(torch.bfloat16)
    return q.to(DEV), k.to(DEV), v.to(DEV)


def check(out, lse, ref):
    o, l, ro, rl = f64(out), f64(lse), ref["out"], ref["lse"]
    np.testing.assert_allclose(o, ro, rtol=1e-4, atol=2e-5)
    fin = np.isfinite(rl)
    np.testing.assert_array_equal(np.isfinite(l), fin)
    assert np.all(l[~fin] == -np.inf)
    np.testing.assert_allclose(l[fin], rl[fin], rtol=0, atol=1e-4)


@pytest.mark.parametrize("layers,H,Hkv,lens,scale", [
    (1, 4, 2, [300, 1, 129, 128, 700], 1.0),      # GQA, a one-row sequence, tile edges
    (2, 2, 2, [1000], 1.0),                        # layers, one long sequence
    (1, 3, 1, [257, 5], 2.5),                      # peaked softmax (larger logits)
])
def test_row_order_against_the_oracle(layers, H, Hkv, lens, scale):
    offs = [0] + list(np.cumsum(lens))
    q, k, v = inputs(layers, offs[-1], H, Hkv, 11 + len(lens), scale)
    out, lse = api().kvsel_reverse_attention(q, k, v, offs)
    assert_ok()
    check(out, lse, oracle.reverse_packed(f64(q), f64(k), f64(v), offs))
    # the last row of every sequence: no future
    for b in range(len(lens)):
        last = offs[b + 1] - 1
        assert torch.all(out[:, last] == 0)
        assert torch.all(lse[:, :, last] == float("-inf"))


def test_explicit_positions_follow_the_rows():
    """A refresh reorders the memory: rows permuted within each sequence, their
    original positions passed; every key tile is visited."""
    lens = [400, 130]
    offs = [0, 400, 530]
    q, k, v = inputs(1, 530, 4, 4, 21)
    gen = np.random.default_rng(22)
    pos = np.concatenate([gen.permutation(400), gen.permutation(130)]).astype(np.int32)
    pos_t = torch.tensor(pos, device=DEV)
    out, lse = api().kvsel_reverse_attention(q, k, v, offs, positions=pos_t)
    assert_ok()
    check(out, lse, oracle.reverse_packed(f64(q), f64(k), f64(v), offs, positions=pos))
    # the same rows in position order give the same results, moved
    order = np.concatenate([np.argsort(pos[:400]), 400 + np.argsort(pos[400:])])
    o_t = torch.tensor(order, device=DEV)
    out2, lse2 = api().kvsel_reverse_attention(q[:, o_t].contiguous(), k[:, o_t].contiguous(),
                                               v[:, o_t].contiguous(), offs)
    assert_ok()
    # fp32 sums over the key tiles in another order: the oracle's bar
    torch.testing.assert_close(out2, out[:, o_t], rtol=1e-4, atol=2e-5)
    fin = torch.isfinite(lse2)
    torch.testing.assert_close(lse2[fin], lse[:, :, o_t][fin], rtol=0, atol=1e-4)
    assert len(lens) == 2


def test_full_size_sampled_rows():
    """One layer, 28 query heads over 4 K/V heads, n = 4096 (the page's larger
    cache): sampled rows of three heads against the decode oracle over their
    future rows; structure everywhere."""
    n = 4096
    q, k, v = inputs(1, n, 28, 4, 31)
    out, lse = api().kvsel_reverse_attention(q, k, v, [0, n])
    assert_ok()
    assert torch.isfinite(out).all()
    assert torch.isfinite(lse[:, :, :n - 1]).all() and torch.all(lse[:, :, n - 1] == float("-inf"))
    q64, k64, v64 = f64(q), f64(k), f64(v)
    rows = np.random.default_rng(32).choice(n - 1, 24, replace=False).tolist() + [0, 127, 128,
                                                                                  4094]
    for h in (0, 13, 27):
        for i in rows:
            o, l = oracle.decode_attention(q64[0, i, h], k64[0, i + 1:, h // 7], v64[0, i + 1:, h // 7])
            np.testing.assert_allclose(f64(out[0, i, h]), o, rtol=1e-4, atol=2e-5)
            assert float(lse[0, h, i]) == pytest.approx(l, abs=1e-4)


def test_nonfinite_key_is_reported():
    q, k, v = inputs(1, 200, 2, 2, 41)
    k[0, 150, 1, 7] = float("inf")
    api().kvsel_reverse_attention(q, k, v, [0, 200])
    assert api().kvsel_device_status() == api().KVSEL_ERR_NONFINITE
    assert api().kvsel_device_status() == 0
