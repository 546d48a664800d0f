"""Jacap scorer on the GPU against the fp64 oracle.

Scores within 1e-4 x the head's largest oracle score (fp32 statistics, the
Gram matrix from bf16 sqrt(w) v products with fp32 accumulation, L^{-1} as a
bf16 hi + lo pair; the oracle reads the same bf16 inputs in fp64); the kept
sets of kvsel_jacap equal the oracle's except at positions whose oracle score
is within that tolerance of the (C - W)-th; gathered rows bit-exact.
"""

import numpy as np
import pytest
import torch

import oracle
from helpers import ensure_built, kept_set_ok
from kv_cache_eviction_snapkv_gb300 import workloads as wk

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
RTOL = 1e-4
TAU, BETA, EPS = 10.0, 0.9, 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def api():
    from kv_cache_eviction_snapkv_gb300 import api as a
    return a


def assert_ok():
    st = api().kvsel_device_status()
    assert st == 0, api().kvsel_status_string(st)


CASES = [
    # name, layers, H, W, C, lens
    ("few_instances_many_splits", 1, 2, 16, 256, [1500, 700, 3000]),
    ("two_layers_window32", 2, 3, 32, 512, [2049, 515]),
    ("short_pool", 1, 2, 8, 64, [200, 136, 9]),
    ("window40_two_query_rounds", 1, 2, 40, 300, [1000, 299]),   # W > 32: queries staged twice
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_scores_and_selection_match_the_oracle(case):
    name, layers, H, W, C, lens = case
    wl = wk.custom_workload(name, layers, H, 128, W, C, "bf16", "avg", 1, lens, 33)
    q, k, v = wk.device_tensors(wl, DEV)
    scores = api().kvsel_jacap_score(q, k, v, wl.offsets, W, TAU, BETA, EPS)
    out_idx, out_k, out_v = api().kvsel_jacap(q, k, v, wl.offsets, W, C, TAU, BETA, EPS)
    assert_ok()
    sc = scores.cpu().numpy()
    idx = out_idx.cpu().numpy()
    n_keep, oo = C - W, 0
    for b, length in enumerate(lens):
        o, n = wl.offsets[b], min(length, C)
        for layer in range(layers):
            for h in range(H):
                qh, kh, vh = wk.head_inputs(wl, layer, b, h)
                got = idx[layer, oo:oo + n, h].tolist()
                if length > W:   # kvsel_jacap_score scores every sequence with a prefix
                    r = oracle.jacap_head(qh, kh, vh, length, TAU, BETA, EPS)["scores"]
                    P = length - W
                    tol = RTOL * r.max()
                    np.testing.assert_allclose(sc[layer, h, o:o + P], r, rtol=0, atol=tol)
                    assert np.all(sc[layer, h, o + P:o + length] == 0)
                if length < C:
                    assert got == list(range(length))
                else:
                    ref = oracle.jacap_head(qh, kh, vh, C, TAU, BETA, EPS)
                    assert got[n_keep:] == list(range(length - W, length))
                    ok, msg = kept_set_ok(got[:n_keep], {"pooled": ref["scores"],
                                                         "indices": ref["indices"]},
                                          n_keep, RTOL * ref["scores"].max())
                    assert ok, f"seq {b} layer {layer} head {h}: {msg}"
                rows = torch.tensor([o + j for j in got], dtype=torch.long, device=DEV)
                assert torch.equal(out_k[layer, oo:oo + n, h], k[layer, rows, h])
                assert torch.equal(out_v[layer, oo:oo + n, h], v[layer, rows, h])
        oo += n


def test_full_size_sampled_heads():
    """32 heads, L = 16384, W = 32, C = 2048: structure everywhere, the oracle on
    two heads."""
    wl = wk.custom_workload("jacap_full", 1, 32, 128, 32, 2048, "bf16", "avg", 1, [16384], 35)
    q, k, v = wk.device_tensors(wl, DEV)
    scores = api().kvsel_jacap_score(q, k, v, wl.offsets, 32, TAU, BETA, EPS)
    out_idx, _, _ = api().kvsel_jacap(q, k, v, wl.offsets, 32, 2048, TAU, BETA, EPS)
    assert_ok()
    sc = scores.cpu().numpy()
    idx = out_idx.cpu().numpy()
    assert np.all(sc[:, :, :16352] > 0) and np.all(np.isfinite(sc))
    for h in (0, 19):
        qh, kh, vh = wk.head_inputs(wl, 0, 0, h)
        ref = oracle.jacap_head(qh, kh, vh, 2048, TAU, BETA, EPS)
        np.testing.assert_allclose(sc[0, h, :16352], ref["scores"], rtol=0,
                                   atol=RTOL * ref["scores"].max())
        ok, msg = kept_set_ok(idx[0, :2016, h].tolist(), {"pooled": ref["scores"],
                                                          "indices": ref["indices"]},
                              2016, RTOL * ref["scores"].max())
        assert ok, msg
