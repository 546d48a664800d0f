"""Full-size parity in the benchmark's launch configuration (one fused
kvsel_snapkv call over the whole workload).

For every named workload:
* sampled (layer, sequence, head) instances against the fp64 oracle: the kept
  prefix set may differ only at positions whose oracle pooled score is within
  1e-4 x (largest vote) of the (C - W)-th largest, the window follows in order,
  and the GPU's score order agrees with the oracle's scores within that
  tolerance;
* every instance: kept prefix positions distinct and inside [0, P), the window
  P..L-1 last, bypass sequences kept whole, and out_K / out_V equal to K / V at
  the output indices (checked on the device with torch indexing).
Plus the all-equal-keys case at the c=0.9 workload's size, where every interior
pooled score ties exactly and the smallest-index rule decides everything.
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


def run_full(wl):
    ensure_built()
    q, k, v = wk.device_tensors(wl, DEV)
    out_idx, out_k, out_v = api().kvsel_snapkv(q, k, v, wl.offsets, wl.window, wl.capacity,
                                               wl.pool_kind, wl.pool_k)
    st = api().kvsel_device_status()
    assert st == 0, api().kvsel_status_string(st)
    return q, k, v, out_idx, out_k, out_v


def check_all_instances(wl, k, v, out_idx, out_k, out_v):
    W, C = wl.window, wl.capacity
    n_keep = C - W
    oo = 0
    for b, length in enumerate(wl.seq_lens):
        n = min(length, C)
        idx = out_idx[:, oo:oo + n, :].long()                    # [layers, n, H]
        if length < C:
            want = torch.arange(length, device=DEV).view(1, -1, 1).expand_as(idx)
            assert torch.equal(idx, want)
        else:
            prefix = length - W
            win = torch.arange(prefix, length, device=DEV).view(1, -1, 1).expand(
                wl.layers, W, wl.heads)
            assert torch.equal(idx[:, n_keep:], win)
            kept = idx[:, :n_keep]
            assert int(kept.min()) >= 0 and int(kept.max()) < prefix
            srt = torch.sort(kept, dim=1).values
            assert bool((srt[:, 1:] != srt[:, :-1]).all()), "duplicate kept positions"
        rows = wl.offsets[b] + idx                                # token rows
        hh = torch.arange(wl.heads, device=DEV).view(1, 1, -1).expand_as(idx)
        ll = torch.arange(wl.layers, device=DEV).view(-1, 1, 1).expand_as(idx)
        assert torch.equal(out_k[:, oo:oo + n], k[ll, rows, hh])
        assert torch.equal(out_v[:, oo:oo + n], v[ll, rows, hh])
        oo += n


def check_sampled(wl, out_idx, samples):
    W, C = wl.window, wl.capacity
    n_keep = C - W
    idx = out_idx.cpu().numpy()
    out_offs = np.concatenate([[0], np.cumsum([min(l, C) for l in wl.seq_lens])])
    ties = []
    for layer, b, h in samples:
        length = wl.seq_lens[b]
        if length < C:
            continue
        qh, kh, vh = wk.head_inputs(wl, layer, b, h)
        ref = oracle.snapkv_head(qh, kh, vh, C, wl.pool_k, wl.pooling)
        oo = out_offs[b]
        got = idx[layer, oo:oo + C, h].tolist()
        assert got[n_keep:] == ref["indices"][n_keep:]
        tol = VOTE_RTOL * ref["votes"].max()
        ok, msg = kept_set_ok(got[:n_keep], ref, n_keep, tol)
        assert ok, f"layer {layer} seq {b} head {h}: {msg}"
        pooled = ref["pooled"][got[:n_keep]]
        assert np.all(pooled[1:] <= pooled[:-1] + tol), "kept positions out of score order"
        kth = np.sort(ref["pooled"])[::-1][n_keep - 1]
        ties.append(int(np.sum(ref["pooled"] == kth)))
    return ties


def _samples(wl, n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        b = int(rng.integers(0, wl.num_seqs))
        out.append((int(rng.integers(0, wl.layers)), b, int(rng.integers(0, wl.heads))))
    return out


@pytest.mark.parametrize("name", ["cfg2", "cfg3", "cfg4", "cfg5"])
def test_full_size_workload(name):
    wl = wk.make_workload(name)
    q, k, v, out_idx, out_k, out_v = run_full(wl)
    check_all_instances(wl, k, v, out_idx, out_k, out_v)
    samples = _samples(wl, 3, 7)
    if name == "cfg4":   # include every sequence, the bypassed one too
        samples = [(0, b, (3 * b) % wl.heads) for b in range(wl.num_seqs)]
    ties = check_sampled(wl, out_idx, samples)
    if name == "cfg5":
        print("exact ties at the budget boundary (sampled heads):", ties)
    del q, k, v, out_idx, out_k, out_v
    torch.cuda.empty_cache()


def test_full_size_all_keys_equal():
    """c=0.9 shape (L=65536, W=16, C=6554, avg 3) with every key equal: each
    prefix vote is H_L - H_P, interior pooled scores tie exactly, the edges
    score 2/3 of that, and the smallest positions win: 1..6538."""
    ensure_built()
    L, W, C, H, D = 65536, 16, 6554, 4, 128
    rng = np.random.default_rng(5)
    q = torch.from_numpy(rng.standard_normal((W, H, D)).astype(np.float32)).to(DEV)
    krow = torch.from_numpy(rng.standard_normal((1, H, D)).astype(np.float32)).to(DEV)
    q = q.to(torch.bfloat16)
    k = krow.to(torch.bfloat16).expand(L, H, D).contiguous()
    v = torch.arange(L, device=DEV, dtype=torch.float32).view(L, 1, 1).expand(L, H, D)
    v = v.to(torch.bfloat16).contiguous()
    out_idx, out_k, out_v = api().kvsel_snapkv(q, k, v, [0, L], W, C, 0, 3)
    assert api().kvsel_device_status() == 0
    n_keep = C - W
    want = list(range(1, n_keep + 1)) + list(range(L - W, L))
    for h in range(H):
        assert out_idx[0, :, h].tolist() == want
    votes, pooled = api().kvsel_score(q, k, [0, L], W, 0, 3)
    s = sum(1.0 / i for i in range(L - W + 1, L + 1))
    vg = votes[0, :, : L - W].float().cpu().numpy()
    np.testing.assert_allclose(vg, s, rtol=1e-4)
    pg = pooled[0, :, : L - W].cpu().numpy()
    assert np.all(pg[:, 1:-1] == pg[:, 1:2])                 # exact ties, bit for bit
