"""kvsel_snapkv_host (cache in host memory) against the device path and the
oracle.

The host path runs the same kernels one layer at a time on q_win and K copied
to the device, with V and the outputs in pinned host memory; its outputs must
be bit-identical to kvsel_snapkv's on the same inputs, and on a ragged case
they are also checked against the fp64 oracle directly: kept prefix sets up
to near-ties at the cut, the window in order, bypass rows whole, and the
gathered rows equal to the host K and V at the output indices.
"""

import ctypes

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


def api():
    from kv_cache_eviction_snapkv_gb300 import api as a
    return a


def assert_ok():
    st = api().kvsel_device_status()
    assert st == 0, api().kvsel_status_string(st)


CASES = [
    # name, layers, H, D, W, C, dtype, pool, k, lens, pin q/K
    ("bf16", 3, 4, 128, 32, 256, "bf16", "avg", 7, [1000, 300, 2600], True),
    ("bf16_pageable_qk", 2, 2, 64, 16, 128, "bf16", "max", 5, [700, 90, 1500], False),
    ("f32", 2, 3, 64, 8, 64, "f32", "avg", 3, [400, 37, 900], True),
    ("bf16_w64_two_pass", 1, 2, 128, 64, 1024, "bf16", "avg", 7, [34000, 2000], True),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_host_path_equals_device_path(case):
    name, layers, H, D, W, C, dtype, pool, kk, lens, pin_qk = case
    wl = wk.custom_workload(name, layers, H, D, W, C, dtype, pool, kk, lens, 77)
    q, k, v = wk.device_tensors(wl, DEV)
    ref = api().kvsel_snapkv(q, k, v, wl.offsets, W, C, wl.pool_kind, kk)
    assert_ok()
    qh = q.cpu().pin_memory() if pin_qk else q.cpu()
    kh = k.cpu().pin_memory() if pin_qk else k.cpu()
    vh = v.cpu().pin_memory()
    stream = torch.cuda.Stream()
    got = api().kvsel_snapkv_host(qh, kh, vh, wl.offsets, W, C, wl.pool_kind, kk, stream=stream)
    stream.synchronize()
    assert_ok()
    for g, r in zip(got, ref):
        assert torch.equal(g, r.cpu())


def test_unpinned_v_or_output_is_rejected():
    a = api()
    wl = wk.custom_workload("host_rules", 1, 2, 64, 8, 32, "bf16", "avg", 3, [200], 3)
    q, k, v = (t.cpu() for t in wk.device_tensors(wl, DEV))
    sh = a.shape_of(k, wl.offsets)
    t_out = a.kvsel_out_tokens(sh, 32)
    oi = torch.empty((1, t_out, 2), dtype=torch.int32, pin_memory=True)
    ok = torch.empty((1, t_out, 2, 64), dtype=torch.bfloat16, pin_memory=True)
    ov = torch.empty_like(ok).pin_memory()
    lib = a._native.lib()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    # V in pageable memory
    assert lib.kvsel_snapkv_host(sh.ref, p(q), p(k), p(v), 8, 32, 0, 3, p(oi), p(ok), p(ov),
                                 None) == a.KVSEL_ERR_INVALID_ARG
    # an output in pageable memory
    vp = v.pin_memory()
    bad = torch.empty((1, t_out, 2, 64), dtype=torch.bfloat16)
    assert lib.kvsel_snapkv_host(sh.ref, p(q), p(k), p(vp), 8, 32, 0, 3, p(oi), p(bad), p(ov),
                                 None) == a.KVSEL_ERR_INVALID_ARG
    # device memory is not host memory
    vd = v.to(DEV)
    assert lib.kvsel_snapkv_host(sh.ref, p(q), p(k), p(vd), 8, 32, 0, 3, p(oi), p(ok), p(ov),
                                 None) == a.KVSEL_ERR_INVALID_ARG
    assert_ok()


def test_host_path_against_oracle():
    a = api()
    wl = wk.custom_workload("host_oracle", 2, 3, 128, 16, 200, "bf16", "avg", 5,
                            [1500, 90, 2700, 200], 91)
    qh, kh, vh = (wk.storage_to_torch(x, wl.dtype) for x in wk.host_tensors(wl))
    qh, kh, vh = qh.pin_memory(), kh.pin_memory(), vh.pin_memory()
    stream = torch.cuda.Stream()
    oi, ok_, ov = a.kvsel_snapkv_host(qh, kh, vh, wl.offsets, wl.window, wl.capacity,
                                      wl.pool_kind, wl.pool_k, stream=stream)
    stream.synchronize()
    assert_ok()
    n_keep = wl.capacity - wl.window
    idx = oi.numpy()
    oo = 0
    for b, length in enumerate(wl.seq_lens):
        n = min(length, wl.capacity)
        o = wl.offsets[b]
        for layer in range(wl.layers):
            for h in range(wl.heads):
                q, k, v = wk.head_inputs(wl, layer, b, h)
                ref = oracle.snapkv_head(q, k, v, wl.capacity, wl.pool_k, wl.pooling)
                got = idx[layer, oo:oo + n, h].tolist()
                if length < wl.capacity:
                    assert got == ref["indices"]
                else:
                    assert got[n_keep:] == ref["indices"][n_keep:]
                    tol = VOTE_RTOL * ref["votes"].max()
                    good, msg = kept_set_ok(got[:n_keep], ref, n_keep, tol)
                    assert good, f"layer {layer} seq {b} head {h}: {msg}"
                rows = torch.tensor([o + j for j in got])
                assert torch.equal(ok_[layer, oo:oo + n, h], kh[layer, rows, h])
                assert torch.equal(ov[layer, oo:oo + n, h], vh[layer, rows, h])
        oo += n
