"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Bars (per head instance):
* window logits within 1e-4 absolute (inputs ~N(0,1), logits O(1..10));
* votes and pooled scores within 1e-4 x the head's largest oracle vote;
* select / compact bit-exact when select is fed the oracle's pooled scores
  rounded to fp32 (the oracle re-runs its selection on those fp32 values);
* end to end: kept prefix sets equal except at positions whose oracle pooled
  score is within that tolerance of the (C - W)-th largest; window appended
  in order; bypass rows 0..L-1; gathered K/V equal to K[idx], V[idx] exactly.
"""

import numpy as np
import pytest
import torch

import oracle
from helpers import VOTE_RTOL, ensure_built, kept_set_ok
from kv_cache_eviction_snapkv_gb300 import workloads as wk

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    from kv_cache_eviction_snapkv_gb300 import api
    api.kvsel_device_status()


def api():
    from kv_cache_eviction_snapkv_gb300 import api as a
    return a


def to_dev(wl):
    q, k, v = wk.host_tensors(wl)
    return tuple(wk.storage_to_torch(x, wl.dtype).to(DEV) for x in (q, k, v))


def assert_ok():
    st = api().kvsel_device_status()
    assert st == 0, api().kvsel_status_string(st)


SCORE_CASES = [
    # name, layers, H, D, W, dtype, pool, k, lens
    ("tc_w32_d128", 2, 3, 128, 32, "bf16", "avg", 7, [700, 32, 2500, 129]),
    ("tc_w16_d128", 1, 2, 128, 16, "bf16", "avg", 3, [4100, 16, 17]),
    ("tc_w64_d128", 1, 2, 128, 64, "bf16", "max", 5, [1200, 64, 1100]),
    ("tc_w5_d64", 1, 3, 64, 5, "bf16", "avg", 1, [300, 5, 2049]),
    ("tc_w1_d64", 1, 2, 64, 1, "bf16", "max", 3, [260, 1]),
    ("tc_w40_d64", 2, 2, 64, 40, "bf16", "avg", 9, [1500, 77]),
    ("gen_f32_d64", 1, 4, 64, 32, "f32", "avg", 7, [1024, 33]),
    ("gen_bf16_d96", 1, 2, 96, 8, "bf16", "avg", 3, [600, 8]),
    ("gen_w80_d128", 1, 2, 128, 80, "bf16", "avg", 5, [900]),
    # long prompts (more than 64 work items per instance): the two-pass kernel,
    # statistics first, then votes from recomputed logits
    ("tc2_w64_d128", 1, 2, 128, 64, "bf16", "avg", 7, [40000, 64, 1500]),
    ("tc2_w40_d64", 1, 2, 64, 40, "bf16", "max", 5, [33500, 40]),
    ("tc2_w32_d128", 2, 2, 128, 32, "bf16", "avg", 7, [70000, 5000, 32, 66000]),
    ("tc2_w16_d64", 1, 3, 64, 16, "bf16", "max", 3, [140000, 16]),
    ("tc2_w5_d128", 1, 2, 128, 5, "bf16", "avg", 1, [139000, 2049]),
]


def _wl(name, layers, H, D, W, dtype, pool, k, lens, seed=5):
    return wk.custom_workload(name, layers, H, D, W, 4 * W + 7, dtype, pool, k, lens, seed)


@pytest.mark.parametrize("case", SCORE_CASES, ids=[c[0] for c in SCORE_CASES])
def test_window_logits(case):
    wl = _wl(*case)
    q, k, _ = to_dev(wl)
    logits = api().kvsel_window_logits(q, k, wl.offsets, wl.window)
    assert_ok()
    lg = logits.cpu().numpy()
    for layer in range(wl.layers):
        for b, length in enumerate(wl.seq_lens):
            o = wl.offsets[b]
            for h in range(wl.heads):
                qh, kh, _ = wk.head_inputs(wl, layer, b, h)
                z = oracle.window_logits(qh, kh)
                np.testing.assert_allclose(lg[layer, h, :, o:o + length], z, atol=1e-4, rtol=1e-5)


@pytest.mark.parametrize("case", SCORE_CASES, ids=[c[0] for c in SCORE_CASES])
def test_votes_and_pooled(case):
    wl = _wl(*case)
    q, k, _ = to_dev(wl)
    votes, pooled = api().kvsel_score(q, k, wl.offsets, wl.window, wl.pool_kind, wl.pool_k)
    assert_ok()
    vg, pg = votes.cpu().numpy(), pooled.cpu().numpy()
    for layer in range(wl.layers):
        for b, length in enumerate(wl.seq_lens):
            o = wl.offsets[b]
            prefix = length - wl.window
            for h in range(wl.heads):
                qh, kh, vh = wk.head_inputs(wl, layer, b, h)
                if length == wl.window:          # no prefix: nothing to vote for
                    assert np.all(vg[layer, h, o:o + length] == 0)
                    continue
                # capacity = L runs the oracle's normal (scoring) path
                ref = oracle.snapkv_head(qh, kh, vh, length, wl.pool_k, wl.pooling)
                tol = VOTE_RTOL * ref["votes"].max()
                np.testing.assert_allclose(vg[layer, h, o:o + prefix], ref["votes"], atol=tol, rtol=0)
                np.testing.assert_allclose(pg[layer, h, o:o + prefix], ref["pooled"], atol=tol, rtol=0)
                assert np.all(vg[layer, h, o + prefix:o + length] == 0)
                assert np.all(pg[layer, h, o + prefix:o + length] == 0)


def test_score_path_choice():
    a = api()
    sh = a.Shape(1, 4, 128, a.KVSEL_BF16, [0, 5000])
    assert a.kvsel_score_path(sh, 32, 0) == 1
    assert a.kvsel_score_path(sh, 64, 1024) == 1
    assert a.kvsel_score_path(sh, 65, 1024) == 0
    assert a.kvsel_score_path(a.Shape(1, 4, 128, a.KVSEL_BF16, [0, 40000]), 64, 1024) == 3
    assert a.kvsel_score_path(a.Shape(1, 4, 128, a.KVSEL_BF16, [0, 70000]), 32, 1024) == 3
    assert a.kvsel_score_path(a.Shape(1, 4, 128, a.KVSEL_BF16, [0, 65536]), 32, 1024) == 1
    assert a.kvsel_score_path(a.Shape(1, 4, 128, a.KVSEL_BF16, [0, 32768]), 64, 1024) == 1
    assert a.kvsel_score_path(a.Shape(1, 4, 64, a.KVSEL_F32, [0, 5000]), 32, 0) == 0
    assert a.kvsel_score_path(a.Shape(1, 4, 96, a.KVSEL_BF16, [0, 5000]), 32, 0) == 0


def _pooled_from_oracle(wl):
    """Oracle pooled scores rounded to fp32, laid out [layers, H, T], + refs."""
    pooled = np.zeros((wl.layers, wl.heads, wl.total), np.float32)
    for layer in range(wl.layers):
        for b, length in enumerate(wl.seq_lens):
            if length < wl.capacity:
                continue
            o = wl.offsets[b]
            for h in range(wl.heads):
                qh, kh, vh = wk.head_inputs(wl, layer, b, h)
                ref = oracle.snapkv_head(qh, kh, vh, wl.capacity, wl.pool_k, wl.pooling)
                pooled[layer, h, o:o + length - wl.window] = ref["pooled"].astype(np.float32)
    return pooled


SELECT_CASES = [
    ("small", 2, 3, 64, 8, "bf16", "avg", 3, [200, 40, 57, 1000]),
    ("k1", 1, 2, 64, 4, "bf16", "max", 5, [300, 5]),
    ("L_eq_C", 1, 2, 64, 16, "bf16", "avg", 7, [71, 300]),
]


@pytest.mark.parametrize("case", SELECT_CASES, ids=[c[0] for c in SELECT_CASES])
def test_select_bitexact_on_oracle_pooled(case):
    name, layers, H, D, W, dtype, pool, kk, lens = case
    C = {"small": 60, "k1": 5, "L_eq_C": 71}[name]
    wl = wk.custom_workload(name, layers, H, D, W, C, dtype, pool, kk, lens, 9)
    pooled = _pooled_from_oracle(wl)
    idx = api().kvsel_select(torch.from_numpy(pooled).to(DEV), wl.offsets, H, W, C)
    assert_ok()
    got = idx.cpu().numpy()
    oo = 0
    for b, length in enumerate(wl.seq_lens):
        n = min(length, C)
        for layer in range(layers):
            for h in range(H):
                o = wl.offsets[b]
                want = oracle.select_from_pooled(
                    pooled[layer, h, o:o + max(0, length - W)].astype(np.float64), length, W, C)
                assert got[layer, oo:oo + n, h].tolist() == want
        oo += n


def test_select_ties_and_nan():
    """Massive exact ties resolve to the smaller position; -0 == +0; NaN ranks last
    and raises NONFINITE."""
    a = api()
    rng = np.random.default_rng(3)
    H, W, C = 4, 8, 520
    lens = [5000, 3000]
    offs = [0, 5000, 8000]
    pooled = rng.choice(np.array([0.0, 0.25, 0.5, 1.0, 2.0], np.float32),
                        size=(1, H, 8000)).astype(np.float32)
    pooled[0, 1, :100] = -0.0
    idx = a.kvsel_select(torch.from_numpy(pooled).to(DEV), offs, H, W, C)
    assert_ok()
    got = idx.cpu().numpy()
    oo = 0
    for b, length in enumerate(lens):
        for h in range(H):
            o = offs[b]
            want = oracle.select_from_pooled(pooled[0, h, o:o + length - W].astype(np.float64),
                                             length, W, C)
            assert got[0, oo:oo + C, h].tolist() == want
        oo += C
    pooled[0, 2, 7] = np.nan
    idx = a.kvsel_select(torch.from_numpy(pooled).to(DEV), offs, H, W, C)
    assert a.kvsel_device_status() == a.KVSEL_ERR_NONFINITE
    assert 7 not in idx.cpu().numpy()[0, :C - W, 2].tolist()


def test_select_largest_budget():
    """C - W = 16384 (the on-chip sort limit) on a 40000-token prompt."""
    a = api()
    rng = np.random.default_rng(4)
    W, C, L = 16, 16400, 40000
    pooled = (rng.random((1, 2, L)) * 1e-3).astype(np.float32)
    pooled[0, 0, ::7] = pooled[0, 0, 3]          # exact ties
    idx = a.kvsel_select(torch.from_numpy(pooled).to(DEV), [0, L], 2, W, C)
    assert_ok()
    got = idx.cpu().numpy()
    for h in range(2):
        want = oracle.select_from_pooled(pooled[0, h, :L - W].astype(np.float64), L, W, C)
        assert got[0, :, h].tolist() == want


def test_select_packed_ragged_batch():
    """A ragged batch whose longest prefix needs 3-CTA clusters: the two long
    sequences take whole clusters, the short one and the bypass one run one per
    CTA of a packed cluster; every instance bit-exact against the oracle."""
    a = api()
    rng = np.random.default_rng(6)
    H, W, C = 3, 16, 2000
    lens = [40000, 3000, 20, 17000]
    offs = [0] + [int(x) for x in np.cumsum(lens)]
    pooled = (rng.random((1, H, offs[-1])) * 1e-3).astype(np.float32)
    pooled[0, 1, ::5] = pooled[0, 1, 2]          # exact ties
    idx = a.kvsel_select(torch.from_numpy(pooled).to(DEV), offs, H, W, C)
    assert_ok()
    got = idx.cpu().numpy()
    oo = 0
    for b, length in enumerate(lens):
        n = min(length, C)
        for h in range(H):
            if length < C:
                assert got[0, oo:oo + n, h].tolist() == list(range(length))
            else:
                o = offs[b]
                want = oracle.select_from_pooled(
                    pooled[0, h, o:o + length - W].astype(np.float64), length, W, C)
                assert got[0, oo:oo + n, h].tolist() == want
        oo += n


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f32", 64), ("f32", 2), ("bf16", 3)])
def test_compact_bitexact(dtype, D):
    a = api()
    wl = wk.custom_workload("c", 2, 3, D, 4, 50, dtype, "avg", 3, [120, 30, 50, 77], 11)
    q, k, v = to_dev(wl)
    rng = np.random.default_rng(1)
    t_out = wl.out_tokens
    idx = np.zeros((2, t_out, 3), np.int32)
    oo = 0
    for length in wl.seq_lens:
        n = min(length, wl.capacity)
        for layer in range(2):
            for h in range(3):
                idx[layer, oo:oo + n, h] = rng.permutation(length)[:n]
        oo += n
    out_k, out_v = a.kvsel_compact(k, v, wl.offsets, torch.from_numpy(idx).to(DEV), wl.capacity)
    assert_ok()
    kh, vh = k.cpu(), v.cpu()
    oo = 0
    for b, length in enumerate(wl.seq_lens):
        n = min(length, wl.capacity)
        for layer in range(2):
            for h in range(3):
                rows = torch.from_numpy(wl.offsets[b] + idx[layer, oo:oo + n, h].astype(np.int64))
                assert torch.equal(out_k[layer, oo:oo + n, h].cpu(), kh[layer, rows, h])
                assert torch.equal(out_v[layer, oo:oo + n, h].cpu(), vh[layer, rows, h])
        oo += n


def test_compact_bad_index_is_reported_not_read():
    a = api()
    wl = wk.custom_workload("c", 1, 2, 64, 4, 16, "bf16", "avg", 3, [40, 20], 12)
    q, k, v = to_dev(wl)
    idx = torch.zeros((1, wl.out_tokens, 2), dtype=torch.int32)
    idx[0, 3, 1] = 40            # == L of sequence 0: out of range
    idx[0, 20, 0] = -1
    a.kvsel_compact(k, v, wl.offsets, idx.to(DEV), wl.capacity)
    assert a.kvsel_device_status() == a.KVSEL_ERR_BAD_INDEX
    assert a.kvsel_device_status() == a.KVSEL_OK          # cleared by the read


E2E_CASES = [
    ("bf16_tc", 2, 4, 128, 32, 256, "bf16", "avg", 7, [3000, 200, 256, 1031]),
    ("bf16_tc_w16_max", 1, 3, 64, 16, 100, "bf16", "max", 5, [2000, 99, 640]),
    ("f32_generic", 1, 4, 64, 32, 256, "f32", "avg", 7, [1024]),
    ("bf16_tc_w64", 1, 2, 128, 64, 300, "bf16", "avg", 3, [5000, 64, 65]),
    ("bf16_tc_w64_two_pass", 1, 2, 128, 64, 2048, "bf16", "avg", 7, [36000, 3000, 2047]),
    # every sequence shorter than C: no scoring launch, the selection (a programmatic
    # dependent launch) follows the set-up copies directly
    ("all_bypass", 2, 3, 64, 16, 256, "bf16", "avg", 7, [100, 37, 255]),
]


@pytest.mark.parametrize("case", E2E_CASES, ids=[c[0] for c in E2E_CASES])
def test_snapkv_end_to_end(case):
    name, layers, H, D, W, C, dtype, pool, kk, lens = case
    wl = wk.custom_workload(name, layers, H, D, W, C, dtype, pool, kk, lens, 21)
    q, k, v = to_dev(wl)
    out_idx, out_k, out_v = api().kvsel_snapkv(q, k, v, wl.offsets, W, C, wl.pool_kind, kk)
    assert_ok()
    check_end_to_end(wl, out_idx.cpu().numpy(), out_k.cpu(), out_v.cpu(), k.cpu(), v.cpu())


def check_end_to_end(wl, idx, gk, gv, kk, vv, heads=None, layers=None):
    W, C = wl.window, wl.capacity
    n_keep = C - W
    oo = 0
    for b, length in enumerate(wl.seq_lens):
        n = min(length, C)
        for layer in (range(wl.layers) if layers is None else layers):
            for h in (range(wl.heads) if heads is None else heads):
                got = idx[layer, oo:oo + n, h].tolist()
                if length < C:
                    assert got == list(range(length))
                else:
                    qh, kh, vh = wk.head_inputs(wl, layer, b, h)
                    ref = oracle.snapkv_head(qh, kh, vh, C, wl.pool_k, wl.pooling)
                    assert got[n_keep:] == list(range(length - W, length))
                    ok, msg = kept_set_ok(got[:n_keep], ref, n_keep, VOTE_RTOL * ref["votes"].max())
                    assert ok, f"seq {b} layer {layer} head {h}: {msg}"
                rows = torch.tensor([wl.offsets[b] + j for j in got], dtype=torch.long)
                assert torch.equal(gk[layer, oo:oo + n, h], kk[layer, rows, h])
                assert torch.equal(gv[layer, oo:oo + n, h], vv[layer, rows, h])
        oo += n


def test_hand_example_on_gpu(golden_dir):
    """The page's worked example (fp32, D = 2) through the fused path."""
    import json, math, os
    g = json.load(open(os.path.join(golden_dir, "worked_example.json")))["printed_on_page"]
    a_w = [x if x is not None else 1 for x in g["exp_weights_query6"]]
    b_w = g["exp_weights_query7"]
    K = torch.tensor([[math.log(x), math.log(y)] for x, y in zip(a_w, b_w)], dtype=torch.float32)
    V = torch.tensor([[float(j), -float(j)] for j in range(8)], dtype=torch.float32)
    q = torch.tensor([[math.sqrt(2), 0.0], [0.0, math.sqrt(2)]], dtype=torch.float32)
    a = api()
    idx, ok, ov = a.kvsel_snapkv(q.view(2, 1, 2).to(DEV), K.view(8, 1, 2).to(DEV),
                                 V.view(8, 1, 2).to(DEV), [0, 8], 2, 5, a.KVSEL_POOL_AVG, 3)
    assert_ok()
    assert idx.cpu().view(-1).tolist() == g["indices"]
    assert torch.equal(ov.cpu().view(5, 2), V[g["indices"]])
    votes, pooled = a.kvsel_score(q.view(2, 1, 2).to(DEV), K.view(8, 1, 2).to(DEV), [0, 8], 2,
                                  a.KVSEL_POOL_AVG, 3)
    want = [51 / 650, 77 / 650, 46 / 65, 254 / 325, 51 / 650, 51 / 650]
    np.testing.assert_allclose(votes.cpu().view(-1)[:6].numpy(), want, rtol=1e-5)


def test_all_bypass_and_single_token_window():
    a = api()
    wl = wk.custom_workload("byp", 1, 2, 128, 1, 64, "bf16", "avg", 1, [63, 1, 20], 2)
    q, k, v = to_dev(wl)
    idx, ok_, ov = a.kvsel_snapkv(q, k, v, wl.offsets, 1, 64, 0, 1)
    assert_ok()
    check_end_to_end(wl, idx.cpu().numpy(), ok_.cpu(), ov.cpu(), k.cpu(), v.cpu())


def test_pool_wider_than_prefix_and_L_equal_C():
    a = api()
    wl = wk.custom_workload("wide", 1, 2, 64, 8, 14, "bf16", "avg", 31, [14, 300], 3)
    q, k, v = to_dev(wl)
    idx, ok_, ov = a.kvsel_snapkv(q, k, v, wl.offsets, 8, 14, 0, 31)
    assert_ok()
    check_end_to_end(wl, idx.cpu().numpy(), ok_.cpu(), ov.cpu(), k.cpu(), v.cpu())


def test_nonfinite_key_is_reported():
    a = api()
    wl = wk.custom_workload("nf", 1, 2, 128, 16, 64, "bf16", "avg", 3, [500], 4)
    q, k, v = to_dev(wl)
    k[0, 123, 1, 5] = float("inf")
    a.kvsel_snapkv(q, k, v, wl.offsets, 16, 64, 0, 3)
    assert a.kvsel_device_status() == a.KVSEL_ERR_NONFINITE
    k[0, 123, 1, 5] = float("nan")
    q32 = q.float()
    a.kvsel_score(q32, k.float(), wl.offsets, 16, 0, 3)
    assert a.kvsel_device_status() == a.KVSEL_ERR_NONFINITE


def test_bounded_wait_reports_timeout():
    """A withheld row-statistics publication makes the other chunks of that
    instance wait until the (short) limit; the kernel reports TIMEOUT and
    exits, and the context stays usable."""
    a = api()
    wl = wk.custom_workload("to", 1, 2, 128, 32, 256, "bf16", "avg", 7, [9000], 6)
    q, k, v = to_dev(wl)
    a.kvsel_set_wait_limit_ns(20_000_000)
    try:
        a.kvsel_debug_inject(1)
        a.kvsel_snapkv(q, k, v, wl.offsets, 32, 256, 0, 7)
        assert a.kvsel_device_status() == a.KVSEL_ERR_TIMEOUT
    finally:
        a.kvsel_debug_inject(0)
        a.kvsel_set_wait_limit_ns(2_000_000_000)
    idx, ok_, ov = a.kvsel_snapkv(q, k, v, wl.offsets, 32, 256, 0, 7)
    assert_ok()
    check_end_to_end(wl, idx.cpu().numpy(), ok_.cpu(), ov.cpu(), k.cpu(), v.cpu())
