"""Pins for the Jacap oracle (weights, capacity matrix, leverage, selection).

Each pin comes from outside the leverage code path (Cholesky + triangular
solve): the page's worked example (tests/golden/jacap_example.json), the
matrix determinant lemma (r_i = 1 - det(A without i) / det(A), by numpy's
slogdet), the trace identity sum_i r_i = d - tr(A^{-1}), closed forms of the
weights at tau -> infinity and of kappa at Lambda = I, the small-w limit
r_i -> w_i |u_i|^2, and the running statistics at beta = 0 and for constant
queries.
"""

import json
import os

import numpy as np
import pytest

import oracle.jacap_oracle as jc
from oracle.snapkv_oracle import OracleArgumentError

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "jacap_example.json")


def test_page_worked_example():
    g = json.load(open(GOLDEN))["printed_on_page"]
    u = np.array(g["u"])
    w = np.array(g["w"])
    r = jc.leverage(w, u)["r"]
    # independent weighting ranks 1 and 2 first (1-based on the page)
    assert sorted((np.argsort(-w, kind="stable")[:2] + 1).tolist()) == g["independent_weighting_prefers"]
    # leverage ranks the novel direction (token 3) first; the kept pair spans both axes
    top2 = (np.argsort(-r, kind="stable")[:2] + 1).tolist()
    assert top2[0] == 3 and 3 in top2
    kept = u[np.array(top2) - 1]
    assert abs(np.linalg.det(kept)) > 0.9
    # tokens 1 and 2 share a direction: their leverage is discounted below w
    assert r[0] < 0.5 * w[0] and r[1] < 0.5 * w[1]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_determinant_lemma(seed):
    rng = np.random.default_rng(seed)
    n, d = 30, 5
    u = rng.standard_normal((n, d))
    w = rng.uniform(0.0, 2.0, n)
    lev = jc.leverage(w, u)
    _, logdet = np.linalg.slogdet(lev["A"])
    for i in range(n):
        _, logdet_wo = np.linalg.slogdet(lev["A"] - w[i] * np.outer(u[i], u[i]))
        assert lev["r"][i] == pytest.approx(1.0 - np.exp(logdet_wo - logdet), rel=1e-10, abs=1e-13)


def test_trace_identity():
    rng = np.random.default_rng(3)
    u = rng.standard_normal((200, 8))
    w = rng.uniform(0, 0.3, 200)
    lev = jc.leverage(w, u)
    assert lev["r"].sum() == pytest.approx(8 - np.trace(np.linalg.inv(lev["A"])), rel=1e-12)


def test_weights_closed_forms():
    rng = np.random.default_rng(4)
    k = rng.standard_normal((50, 6))
    mu = rng.standard_normal(6)
    lam = rng.uniform(0.5, 2, 6)
    wt = jc.weights(k, mu, lam, 1e12)            # tau -> infinity: uniform attention
    np.testing.assert_allclose(wt["alpha"], 1 / 50, rtol=1e-9)
    np.testing.assert_allclose(wt["kappa"], (k * k * lam).sum(axis=1), rtol=1e-14)
    np.testing.assert_allclose(wt["w"], (1 / 50 * 49 / 50) ** 2 * wt["kappa"] / 6, rtol=1e-8)
    wi = jc.weights(k, mu, np.ones(6), 1.0)      # Lambda = I: kappa = |k|^2
    np.testing.assert_allclose(wi["kappa"], np.linalg.norm(k, axis=1) ** 2, rtol=1e-14)
    z = k @ mu / np.sqrt(6)
    np.testing.assert_allclose(wi["alpha"], np.exp(z) / np.exp(z).sum(), rtol=1e-12)


def test_small_weight_limit():
    rng = np.random.default_rng(5)
    u = rng.standard_normal((40, 4))
    w = np.full(40, 1e-9)
    r = jc.leverage(w, u)["r"]
    np.testing.assert_allclose(r, w * np.linalg.norm(u, axis=1) ** 2, rtol=1e-6)


def test_window_statistics():
    q = np.array([[1.0, 2.0], [3.0, -1.0], [0.5, 0.5]])
    mu, lam = jc.window_statistics(q, 0.0, 1e-6)          # beta = 0: the last query
    np.testing.assert_array_equal(mu, q[-1])
    np.testing.assert_array_equal(lam, [1e-6, 1e-6])
    const = np.tile([0.3, -0.7], (5, 1))
    mu, lam = jc.window_statistics(const, 0.9, 1e-4)
    np.testing.assert_allclose(mu, [0.3, -0.7], rtol=1e-15)
    np.testing.assert_allclose(lam, [1e-4, 1e-4])
    mu, lam = jc.window_statistics(q, 0.5, 0.0)           # by hand
    m1 = 0.5 * q[0] + 0.5 * q[1]
    s1 = 0.5 * q[0] ** 2 + 0.5 * q[1] ** 2
    m2 = 0.5 * m1 + 0.5 * q[2]
    s2 = 0.5 * s1 + 0.5 * q[2] ** 2
    np.testing.assert_allclose(mu, m2, rtol=1e-15)
    np.testing.assert_allclose(lam, s2 - m2 * m2, rtol=1e-14)


def test_head_selection_structure():
    rng = np.random.default_rng(6)
    L, W, C, D = 120, 8, 40, 6
    q = rng.standard_normal((W, D))
    k = rng.standard_normal((L, D))
    v = rng.standard_normal((L, D))
    r = jc.jacap_head(q, k, v, C, tau=10.0)
    idx = r["indices"]
    assert idx[C - W:] == list(range(L - W, L))
    kept = idx[:C - W]
    s = r["scores"]
    assert len(set(kept)) == C - W and max(kept) < L - W
    assert min(s[kept]) >= max(np.delete(s, kept))
    assert jc.jacap_head(q[:3], k[:10], v[:10], 20)["indices"] == list(range(10))   # bypass
    with pytest.raises(OracleArgumentError):
        jc.jacap_head(q, k, v, W)


@pytest.mark.parametrize("seed", [3, 4])
def test_leverage_bound_from_sherman_morrison(seed):
    """A >= I + w_i u_i u_i^T, so r_i <= w_i |u_i|^2 / (1 + w_i |u_i|^2) < 1
    (Sherman-Morrison on the rank-one term), with equality for a lone token."""
    rng = np.random.default_rng(seed)
    u = rng.standard_normal((50, 6))
    w = rng.uniform(0.0, 3.0, 50)
    r = jc.leverage(w, u)["r"]
    q = w * np.sum(u * u, axis=1)
    assert np.all(r >= 0.0)
    assert np.all(r <= q / (1.0 + q) * (1 + 1e-12))
    lone = jc.leverage(w[:1], u[:1])["r"][0]
    assert lone == pytest.approx(q[0] / (1.0 + q[0]), rel=1e-12)
