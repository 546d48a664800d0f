"""Grouped-query attention on the GPU against the oracle.

q_win has H query heads and K, V have H_kv = H / G heads. kvsel_snapkv selects
per query head on the K/V head h / G (the expanded reading of the page's GQA
section); kvsel_snapkv_grouped selects once per K/V head on the summed votes of
its G query heads (our reading). Inputs: the query heads come from one seeded
workload with H heads, K and V from another with H_kv heads and the same
sequence lengths.
"""

import numpy as np
import pytest
import torch

import oracle
from helpers import VOTE_RTOL, ensure_built, kept_set_ok
from kv_cache_eviction_snapkv_gb300 import workloads as wk

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def api():
    from kv_cache_eviction_snapkv_gb300 import api as a
    return a


def make(name, layers, hq, hkv, dim, window, capacity, dtype, pooling, pool_k, lens, seed):
    wq = wk.custom_workload(name + "q", layers, hq, dim, window, capacity, dtype, pooling, pool_k,
                            lens, seed)
    wkv = wk.custom_workload(name + "kv", layers, hkv, dim, window, capacity, dtype, pooling,
                             pool_k, lens, seed + 500)
    q, _, _ = wk.device_tensors(wq, DEV)
    _, k, v = wk.device_tensors(wkv, DEV)
    return wq, wkv, q, k, v


def assert_ok():
    st = api().kvsel_device_status()
    assert st == 0, api().kvsel_status_string(st)


def group_inputs(wq, wkv, layer, b, kvh):
    g = wq.heads // wkv.heads
    qs = np.stack([wk.head_inputs(wq, layer, b, kvh * g + j)[0] for j in range(g)])
    _, kh, vh = wk.head_inputs(wkv, layer, b, kvh)
    return qs, kh, vh


CASES = [
    # name, layers, H, H_kv, D, W, C, dtype, pool, k, lens
    ("g4_bf16", 1, 8, 2, 128, 32, 256, "bf16", "avg", 7, [1200, 300, 2600]),
    ("g2_bf16_max", 2, 4, 2, 64, 16, 128, "bf16", "max", 5, [700, 1900]),
    ("g4_f32", 1, 4, 1, 64, 8, 64, "f32", "avg", 3, [400, 37, 900]),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_repeat_mode_matches_oracle(case):
    ensure_built()
    name, layers, hq, hkv, D, W, C, dtype, pool, kk, lens = case
    wq, wkv, q, k, v = make(name, layers, hq, hkv, D, W, C, dtype, pool, kk, lens, 31)
    out_idx, out_k, out_v = api().kvsel_snapkv(q, k, v, wq.offsets, W, C, wq.pool_kind, kk)
    assert_ok()
    assert out_idx.shape[-1] == hq and out_k.shape[2] == hq
    g = hq // hkv
    idx = out_idx.cpu().numpy()
    n_keep, oo = C - W, 0
    for b, length in enumerate(lens):
        n = min(length, C)
        for layer in range(layers):
            for h in range(hq):
                got = idx[layer, oo:oo + n, h].tolist()
                if length < C:
                    assert got == list(range(length))
                else:
                    qh = wk.head_inputs(wq, layer, b, h)[0]
                    _, kh, vh = wk.head_inputs(wkv, layer, b, h // g)
                    ref = oracle.snapkv_head(qh, kh, vh, C, kk, pool)
                    assert got[n_keep:] == list(range(length - W, length))
                    ok, msg = kept_set_ok(got[:n_keep], ref, n_keep,
                                          VOTE_RTOL * ref["votes"].max())
                    assert ok, f"seq {b} layer {layer} head {h}: {msg}"
                rows = torch.tensor([wq.offsets[b] + j for j in got], dtype=torch.long,
                                    device=DEV)
                assert torch.equal(out_k[layer, oo:oo + n, h], k[layer, rows, h // g])
                assert torch.equal(out_v[layer, oo:oo + n, h], v[layer, rows, h // g])
        oo += n


def test_repeat_mode_votes_per_query_head():
    ensure_built()
    wq, wkv, q, k, v = make("votes", 1, 8, 2, 128, 32, 256, "bf16", "avg", 7, [1500, 900], 41)
    votes, pooled = api().kvsel_score(q, k, wq.offsets, 32, wq.pool_kind, 7)
    assert_ok()
    vg = votes.cpu().numpy()
    for b, length in enumerate(wq.seq_lens):
        o = wq.offsets[b]
        for h in range(8):
            qh = wk.head_inputs(wq, 0, b, h)[0]
            _, kh, vh = wk.head_inputs(wkv, 0, b, h // 4)
            ref = oracle.snapkv_head(qh, kh, vh, 256, 7, "avg")
            p = length - 32
            np.testing.assert_allclose(vg[0, h, o:o + p], ref["votes"], rtol=0,
                                       atol=VOTE_RTOL * ref["votes"].max())


# group-shared scoring on the tensor cores (the G query heads of a K/V head as
# G * W <= 64 window rows of one MMA): ragged lengths, bypass, padded rows
GROUP_CASES = CASES + [
    ("g4_w16_d128", 1, 8, 2, 128, 16, 300, "bf16", "avg", 7, [3000, 150, 5100]),
    ("g2_w24_d64", 2, 4, 2, 64, 24, 200, "bf16", "max", 5, [1000, 2333]),
    ("g8_w8_d128", 1, 16, 2, 128, 8, 100, "bf16", "avg", 3, [900, 1700]),
]


@pytest.mark.parametrize("case", GROUP_CASES, ids=[c[0] for c in GROUP_CASES])
def test_grouped_mode_matches_oracle(case):
    ensure_built()
    name, layers, hq, hkv, D, W, C, dtype, pool, kk, lens = case
    wq, wkv, q, k, v = make(name, layers, hq, hkv, D, W, C, dtype, pool, kk, lens, 51)
    out_idx, out_k, out_v = api().kvsel_snapkv_grouped(q, k, v, wq.offsets, W, C,
                                                       wq.pool_kind, kk)
    assert_ok()
    assert out_idx.shape[-1] == hkv and out_k.shape[2] == hkv
    idx = out_idx.cpu().numpy()
    n_keep, oo = C - W, 0
    for b, length in enumerate(lens):
        n = min(length, C)
        for layer in range(layers):
            for h in range(hkv):
                got = idx[layer, oo:oo + n, h].tolist()
                if length < C:
                    assert got == list(range(length))
                else:
                    qs, kh, vh = group_inputs(wq, wkv, layer, b, h)
                    ref = oracle.snapkv_group(qs, kh, vh, C, kk, pool)
                    assert got[n_keep:] == list(range(length - W, length))
                    # each head's votes carry up to 1e-4 x its max: the sum carries the sum
                    tol = VOTE_RTOL * sum(s.max() for s in ref["head_votes"])
                    ok, msg = kept_set_ok(got[:n_keep], ref, n_keep, tol)
                    assert ok, f"seq {b} layer {layer} kv head {h}: {msg}"
                rows = torch.tensor([wq.offsets[b] + j for j in got], dtype=torch.long,
                                    device=DEV)
                assert torch.equal(out_k[layer, oo:oo + n, h], k[layer, rows, h])
                assert torch.equal(out_v[layer, oo:oo + n, h], v[layer, rows, h])
        oo += n


def test_grouped_with_one_head_per_group_is_the_plain_path():
    ensure_built()
    wl = wk.custom_workload("g1", 2, 4, 128, 32, 512, "bf16", "avg", 7, [3000, 200, 1500], 61)
    q, k, v = wk.device_tensors(wl, DEV)
    a = api().kvsel_snapkv(q, k, v, wl.offsets, 32, 512, 0, 7)
    b = api().kvsel_snapkv_grouped(q, k, v, wl.offsets, 32, 512, 0, 7)
    assert_ok()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_compact_expands_kv_heads():
    """kvsel_compact with out_idx over H query heads and K/V over H_kv heads."""
    ensure_built()
    L, T, hq, hkv, D, C = 2, 600, 6, 3, 64, 128
    offs = [0, 250, 600]
    gen = torch.Generator(device="cpu").manual_seed(7)
    K = torch.randn(L, T, hkv, D, generator=gen).to(torch.bfloat16).to(DEV)
    V = torch.randn(L, T, hkv, D, generator=gen).to(torch.bfloat16).to(DEV)
    t_out = 2 * C
    idx = torch.empty(L, t_out, hq, dtype=torch.int32)
    for b, (o0, o1) in enumerate(zip(offs[:-1], offs[1:])):
        for layer in range(L):
            for h in range(hq):
                idx[layer, b * C:(b + 1) * C, h] = torch.randperm(o1 - o0, generator=gen)[:C]
    idx = idx.to(DEV)
    ok, ov = api().kvsel_compact(K, V, offs, idx, C)
    assert_ok()
    for b in range(2):
        rows = offs[b] + idx[:, b * C:(b + 1) * C].long()
        for h in range(hq):
            ll = torch.arange(L, device=DEV).view(-1, 1).expand(L, C)
            assert torch.equal(ok[:, b * C:(b + 1) * C, h], K[ll, rows[:, :, h], h // 2])
            assert torch.equal(ov[:, b * C:(b + 1) * C, h], V[ll, rows[:, :, h], h // 2])


@pytest.mark.parametrize("W", [32, 16])
def test_grouped_full_size_sampled(W):
    """32 query heads on 8 K/V heads, L = 16384, C = 2048 (the 32-layer shape's
    per-layer size; W = 16 puts the four query heads of a group in one MMA):
    structure everywhere, the oracle on sampled groups."""
    ensure_built()
    wq, wkv, q, k, v = make("gfull", 1, 32, 8, 128, W, 2048, "bf16", "avg", 7, [16384], 71)
    out_idx, out_k, out_v = api().kvsel_snapkv_grouped(q, k, v, wq.offsets, W, 2048, 0, 7)
    assert_ok()
    n_keep = 2048 - W
    kept = out_idx[0, :n_keep].long()
    assert int(kept.min()) >= 0 and int(kept.max()) < 16384 - W
    srt = torch.sort(kept, dim=0).values
    assert bool((srt[1:] != srt[:-1]).all())
    idx = out_idx.cpu().numpy()
    for h in (0, 5):
        qs, kh, vh = group_inputs(wq, wkv, 0, 0, h)
        ref = oracle.snapkv_group(qs, kh, vh, 2048, 7, "avg")
        tol = VOTE_RTOL * sum(s.max() for s in ref["head_votes"])
        ok, msg = kept_set_ok(idx[0, :n_keep, h].tolist(), ref, n_keep, tol)
        assert ok, msg
    rows = out_idx[0].long()
    hh = torch.arange(8, device=DEV).view(1, -1).expand_as(rows)
    assert torch.equal(out_k[0], k[0, rows, hh])
    assert torch.equal(out_v[0], v[0, rows, hh])
