"""kvsel_score_static: the scoring entry point for callers that cannot
allocate device memory (it keeps its scratch in a fixed array inside the
library image). It must give the same votes and pooled scores as kvsel_score
on the same inputs, call after call, and refuse work beyond its fixed size.

This file is collected last, so a run that stops at the first failure has
already run every other test; it also passes alone in a fresh process."""

import ctypes

import numpy as np
import pytest
import torch

from helpers import VOTE_RTOL, ensure_built
from kv_cache_eviction_snapkv_gb300 import workloads as wk

pytestmark = pytest.mark.gpu


def _call_static(lib, sh, q, k, W, kind, pk, votes, pooled):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.kvsel_score_static(sh.ref, ctypes.c_void_p(q.data_ptr()),
                                  ctypes.c_void_p(k.data_ptr()), W, kind, pk,
                                  ctypes.c_void_p(votes.data_ptr()),
                                  ctypes.c_void_p(pooled.data_ptr()), stream)


@pytest.mark.parametrize("dtype,D,W,lens", [("bf16", 128, 32, [3000, 40, 2049]),
                                            ("f32", 64, 16, [1500, 17])])
def test_static_scratch_matches_kvsel_score(dtype, D, W, lens):
    ensure_built()
    from kv_cache_eviction_snapkv_gb300 import _native, api
    dev = torch.device("cuda:0")
    wl = wk.custom_workload("static", 2, 3, D, W, 4 * W, dtype, "avg", 5, lens, 31)
    q, k, _ = (wk.storage_to_torch(x, dtype).to(dev) for x in wk.host_tensors(wl))
    ref_votes, ref_pooled = api.kvsel_score(q, k, wl.offsets, W, wl.pool_kind, wl.pool_k)
    assert api.kvsel_device_status() == 0
    lib = _native.lib()
    sh = api.shape_of(k, wl.offsets)
    rv, rp = ref_votes.cpu().numpy(), ref_pooled.cpu().numpy()
    for _ in range(2):   # the array keeps the previous call's contents
        votes = torch.full_like(ref_votes, float("nan"))
        pooled = torch.full_like(ref_pooled, float("nan"))
        assert _call_static(lib, sh, q, k, W, wl.pool_kind, wl.pool_k, votes, pooled) == 0
        assert api.kvsel_device_status() == 0
        v, p = votes.cpu().numpy(), pooled.cpu().numpy()
        for layer in range(wl.layers):
            for h in range(wl.heads):
                tol = VOTE_RTOL * max(rv[layer, h].max(), 1e-30)
                np.testing.assert_allclose(v[layer, h], rv[layer, h], atol=tol, rtol=0)
                np.testing.assert_allclose(p[layer, h], rp[layer, h], atol=tol, rtol=0)


def test_static_scratch_refuses_oversized_calls():
    ensure_built()
    from kv_cache_eviction_snapkv_gb300 import _native, api
    dev = torch.device("cuda:0")
    # 64 layers x 64 heads x 16 chunks x 32 rows x 8 bytes = 16 MiB of slots > 8 MiB
    sh = api.Shape(64, 64, 128, api.KVSEL_BF16, [0, 16384])
    dummy = torch.empty(1024, dtype=torch.bfloat16, device=dev)
    out = torch.empty(16, dtype=torch.float32, device=dev)
    lib = _native.lib()
    assert _call_static(lib, sh, dummy, dummy, 32, 0, 3, out, out) == api.KVSEL_ERR_UNSUPPORTED
