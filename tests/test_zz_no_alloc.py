"""kvsel_score_static: the scoring entry point for callers that cannot
allocate device memory.

Who needs it: code that runs under a memory allocator it must not bypass (a
serving engine's caching pool, a framework that accounts for every byte), or
in a place where cudaMalloc is not allowed. kvsel_score grows a library
workspace with cudaMalloc; kvsel_score_static keeps its scratch in a fixed
8 MiB array inside the library image instead.

The checks run in a fresh child process, so that nothing else has touched
the library first: the static entry point is called before any other entry
point, its votes and pooled scores are compared with the fp64 oracle, two
calls in a row give results within the tolerance of the other GPU tests, the
library holds no workspace afterwards and the free device memory does not
fall across a call with a larger shape. Only then is kvsel_score called and
the static results compared with its results too.

This file is collected last, so a run that stops at the first failure has
already run every other test; the test passes alone and after the others.
"""

import os
import subprocess
import sys
import textwrap

import pytest

from helpers import ROOT, ensure_built

pytestmark = pytest.mark.gpu

_CHILD = textwrap.dedent(r"""
    import sys
    sys.path.insert(0, {root!r})
    sys.path.insert(0, {tests!r})
    import numpy as np
    import torch
    import oracle
    from helpers import VOTE_RTOL
    from kv_cache_eviction_snapkv_gb300 import api, workloads as wk

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)

    def inputs(wl):
        q, k, _ = (wk.storage_to_torch(x, wl.dtype).to(dev) for x in wk.host_tensors(wl))
        return q, k

    def against_oracle(wl, votes, pooled):
        vg, pg = votes.cpu().numpy(), pooled.cpu().numpy()
        for layer in range(wl.layers):
            for b, length in enumerate(wl.seq_lens):
                o, prefix = wl.offsets[b], length - wl.window
                for h in range(wl.heads):
                    if prefix == 0:
                        assert np.all(vg[layer, h, o:o + length] == 0)
                        continue
                    qh, kh, vh = wk.head_inputs(wl, layer, b, h)
                    ref = oracle.snapkv_head(qh, kh, vh, length, wl.pool_k, wl.pooling)
                    tol = VOTE_RTOL * ref["votes"].max()
                    np.testing.assert_allclose(vg[layer, h, o:o + prefix], ref["votes"],
                                               atol=tol, rtol=0)
                    np.testing.assert_allclose(pg[layer, h, o:o + prefix], ref["pooled"],
                                               atol=tol, rtol=0)
                    assert np.all(vg[layer, h, o + prefix:o + length] == 0)
                    assert np.all(pg[layer, h, o + prefix:o + length] == 0)

    def status_ok():
        st = api.kvsel_device_status()
        assert st == 0, api.kvsel_status_string(st)

    # the same kernels (dtype, head dim, window padding) at two sizes, so that
    # the second call loads no kernel code the first did not
    dtype, D, W = {dtype!r}, {D}, {W}
    small = wk.custom_workload("static_a", 1, 2, D, W, 4 * W, dtype, "avg", 5, {lens_a}, 31)
    large = wk.custom_workload("static_b", 2, 3, D, W, 4 * W, dtype, "max", 3, {lens_b}, 32)
    qa, ka = inputs(small)
    qb, kb = inputs(large)
    outs = {{}}
    for name, wl in (("a", small), ("b", large)):
        for rep in range(2):
            outs[name, rep] = (torch.full((wl.layers, wl.heads, wl.total), float("nan"), device=dev),
                               torch.full((wl.layers, wl.heads, wl.total), float("nan"), device=dev))
    sha = api.shape_of(ka, small.offsets)
    shb = api.shape_of(kb, large.offsets)
    assert 0 < api.kvsel_score_static_bytes(sha, W) <= 8 << 20
    assert 0 < api.kvsel_score_static_bytes(shb, W) <= 8 << 20
    torch.cuda.synchronize()

    # first call of the process: looks up the scratch array (and loads the code)
    api.kvsel_score_static(qa, ka, small.offsets, W, small.pool_kind, small.pool_k, *outs["a", 0])
    torch.cuda.synchronize()
    status_ok()
    free0 = torch.cuda.mem_get_info(dev)[0]
    # a larger call, then the small one again: nothing is allocated
    api.kvsel_score_static(qb, kb, large.offsets, W, large.pool_kind, large.pool_k, *outs["b", 0])
    api.kvsel_score_static(qb, kb, large.offsets, W, large.pool_kind, large.pool_k, *outs["b", 1])
    api.kvsel_score_static(qa, ka, small.offsets, W, small.pool_kind, small.pool_k, *outs["a", 1])
    torch.cuda.synchronize()
    status_ok()
    free1 = torch.cuda.mem_get_info(dev)[0]
    assert api.kvsel_workspace_bytes() == 0, "the static path left a workspace"
    assert free0 - free1 < (1 << 20), f"device memory fell by {{free0 - free1}} bytes"

    # against the oracle, both calls of each shape
    for name, wl in (("a", small), ("b", large)):
        for rep in range(2):
            against_oracle(wl, *outs[name, rep])

    # against the allocating entry point (called only now)
    for name, wl, q, k in (("a", small, qa, ka), ("b", large, qb, kb)):
        rv, rp = api.kvsel_score(q, k, wl.offsets, W, wl.pool_kind, wl.pool_k)
        status_ok()
        rv, rp = rv.cpu().numpy(), rp.cpu().numpy()
        for rep in range(2):
            v, p = (t.cpu().numpy() for t in outs[name, rep])
            for layer in range(wl.layers):
                for h in range(wl.heads):
                    tol = VOTE_RTOL * max(float(rv[layer, h].max()), 1e-30)
                    np.testing.assert_allclose(v[layer, h], rv[layer, h], atol=tol, rtol=0)
                    np.testing.assert_allclose(p[layer, h], rp[layer, h], atol=tol, rtol=0)
    assert api.kvsel_workspace_bytes() > 0
    print("static ok", free0, free1)
""")


@pytest.mark.parametrize("dtype,D,W,lens_a,lens_b", [
    ("bf16", 128, 32, [3000, 40, 2049], [5000, 40, 2049, 1500]),
    ("f32", 64, 16, [1500, 17], [2600, 17, 700]),
])
def test_static_scratch_in_fresh_process(dtype, D, W, lens_a, lens_b):
    ensure_built()
    code = _CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), dtype=dtype, D=D, W=W,
                         lens_a=lens_a, lens_b=lens_b)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    assert "static ok" in res.stdout


def test_static_scratch_refuses_oversized_calls():
    ensure_built()
    import torch
    from kv_cache_eviction_snapkv_gb300 import _native, api
    dev = torch.device("cuda:0")
    # 64 layers x 64 heads x 16 chunks x 32 rows x 8 bytes = 16 MiB of slots > 8 MiB
    sh = api.Shape(64, 64, 128, api.KVSEL_BF16, [0, 16384])
    assert api.kvsel_score_static_bytes(sh, 32) > 8 << 20
    dummy = torch.empty(1024, dtype=torch.bfloat16, device=dev)
    out = torch.empty(16, dtype=torch.float32, device=dev)
    import ctypes
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    assert _native.lib().kvsel_score_static(sh.ref, p(dummy), p(dummy), 32, 0, 3, p(out),
                                            p(out), stream) == api.KVSEL_ERR_UNSUPPORTED
