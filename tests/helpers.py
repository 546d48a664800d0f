"""Shared test helpers: build-once, oracle comparisons and tolerances."""

from __future__ import annotations

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

VOTE_RTOL = 1e-4      # votes and pooled: |gpu - oracle| <= 1e-4 * max oracle vote of the head


def ensure_built():
    from kv_cache_eviction_snapkv_gb300 import build
    return build.build()


def kept_set_ok(got_prefix, ref, n_keep, tol):
    """GPU kept prefix set vs the oracle's: they may differ only at positions whose
    oracle pooled score is within tol of the n_keep-th largest score."""
    pooled = ref["pooled"]
    if len(set(got_prefix)) != n_keep:
        return False, "duplicate or missing kept positions"
    kth = np.sort(pooled)[::-1][n_keep - 1]
    diff = set(got_prefix) ^ set(ref["indices"][:n_keep])
    bad = [j for j in diff if abs(pooled[j] - kth) > tol]
    return (not bad), f"positions differ beyond tolerance: {sorted(bad)[:10]}"
