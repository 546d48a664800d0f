"""Jacap leverage scorer: plain fp64 CPU oracle.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` may import it; the CUDA library
shares nothing with it.

Source: the pages "Jacap reading notes" / "Jacap technical review"
(zhongzhuzhou.org), sections 6 (practical approximation: full-pool attention,
diagonal sensitivity and query response, capacity matrix and leverage score),
7 (Algorithm 1, one eviction event; 7.1 why leverage follows from capacity;
7.2 worked miniature example) and 11 (Algorithm 2, the running mean and
diagonal second moment of the queries):

1. z_i = k_i . mu_Q / (tau sqrt(d_k)); alpha_bar = softmax(z) over the pool;
2. kappa_i = k_i^T Lambda_Q k_i (Lambda_Q diagonal);
3. w_i = [alpha_bar_i (1 - alpha_bar_i)]^2 kappa_i / d_k;
4. u_i = v_i (the value as the output proxy, no W_O);
5. A = I + sum_i w_i u_i u_i^T; factor A once (Cholesky), solve A x_i = u_i;
6. r_i = w_i u_i^T x_i; keep the top B after reserving the protected tokens.
Statistics (Algorithm 2): mu <- beta mu + (1 - beta) q, m <- beta m +
(1 - beta) q * q, diag(Lambda_Q) = max(m - mu * mu, eps).

Readings (ours, where the pages leave it open): in a prompt-time selection
like SnapKV's, the candidate pool is the prefix (positions 0 .. L - W - 1),
the last W tokens are the reserved window, and mu_Q, Lambda_Q come from the W
window queries by Algorithm 2's recursion started from the first window query
(mu = q_0, m = q_0 * q_0); the top C - W scores are kept, ties to the smaller
position, then the window, as in the selection oracle.

Parity status: pinned by ``tests/test_oracle_jacap.py`` (the page's worked
example, the determinant-lemma identity, the trace identity sum_i r_i =
d - tr(A^{-1}), a brute-force inverse, the tau -> infinity and w scaling
limits).
"""

from __future__ import annotations

from typing import Dict, List

import numpy as np

from .snapkv_oracle import OracleArgumentError, top_prefix


def window_statistics(q_win, beta: float, eps: float):
    """(mu_Q, diag Lambda_Q) from the window queries (W, D) by the running
    mean and second moment, started from the first query."""
    q_win = np.asarray(q_win, np.float64)
    if q_win.ndim != 2 or q_win.shape[0] < 1:
        raise OracleArgumentError("q_win must be (W >= 1, D)")
    if not 0.0 <= beta < 1.0 or eps < 0.0:
        raise OracleArgumentError("0 <= beta < 1 and eps >= 0")
    mu = q_win[0].copy()
    m = q_win[0] * q_win[0]
    for q in q_win[1:]:
        mu = beta * mu + (1.0 - beta) * q
        m = beta * m + (1.0 - beta) * q * q
    return mu, np.maximum(m - mu * mu, eps)


def weights(keys, mu_q, lam_q, tau: float) -> Dict[str, np.ndarray]:
    """z, alpha_bar, kappa and w for every candidate key (N, D)."""
    keys = np.asarray(keys, np.float64)
    mu_q = np.asarray(mu_q, np.float64)
    lam_q = np.asarray(lam_q, np.float64)
    if keys.ndim != 2 or keys.shape[0] < 1 or keys.shape[1] != mu_q.shape[0]:
        raise OracleArgumentError("keys must be (N >= 1, D)")
    if tau <= 0:
        raise OracleArgumentError("tau must be positive")
    d = keys.shape[1]
    z = keys @ mu_q / (tau * np.sqrt(d))
    e = np.exp(z - z.max())
    alpha = e / e.sum()
    kappa = (keys * keys) @ lam_q
    w = (alpha * (1.0 - alpha)) ** 2 * kappa / d
    return {"z": z, "alpha": alpha, "kappa": kappa, "w": w}


def capacity_matrix(w, u) -> np.ndarray:
    """A = I + sum_i w_i u_i u_i^T."""
    u = np.asarray(u, np.float64)
    return np.eye(u.shape[1]) + (u * np.asarray(w, np.float64)[:, None]).T @ u


def leverage(w, u) -> Dict[str, np.ndarray]:
    """r_i = w_i u_i^T A^{-1} u_i through one Cholesky factor of A (a library
    factorisation and triangular solves as steps)."""
    w = np.asarray(w, np.float64)
    u = np.asarray(u, np.float64)
    a = capacity_matrix(w, u)
    chol = np.linalg.cholesky(a)                    # A = L L^T
    y = np.linalg.solve(chol, u.T)                  # L y_i = u_i
    r = w * np.sum(y * y, axis=0)                   # u^T A^{-1} u = |L^{-1} u|^2
    return {"A": a, "L": chol, "r": r}


def jacap_head(q_win, keys, values, capacity: int, tau: float = 10.0, beta: float = 0.9,
               eps: float = 1e-6) -> Dict[str, object]:
    """One (layer, sequence, head): Jacap scores of the prefix and the kept
    positions (top C - W by (-r, j), then the window; 0 .. L-1 when L < C)."""
    q_win = np.asarray(q_win, np.float64)
    keys = np.asarray(keys, np.float64)
    values = np.asarray(values, np.float64)
    length, window = keys.shape[0], q_win.shape[0]
    if values.shape != keys.shape:
        raise OracleArgumentError("values must match keys")
    if window < 1 or window > length or capacity <= window:
        raise OracleArgumentError("1 <= W <= L and C > W")
    if length < capacity:
        return {"indices": list(range(length)), "scores": np.zeros(0)}
    prefix = length - window
    mu, lam = window_statistics(q_win, beta, eps)
    wt = weights(keys[:prefix], mu, lam, tau)
    lev = leverage(wt["w"], values[:prefix])
    idx: List[int] = top_prefix(lev["r"], capacity - window) + list(range(prefix, length))
    return {"indices": idx, "scores": lev["r"], "w": wt["w"], "alpha": wt["alpha"],
            "kappa": wt["kappa"], "mu": mu, "lam": lam, "A": lev["A"]}
