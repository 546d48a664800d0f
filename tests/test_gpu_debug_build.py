"""The debug library (-DKVSEL_DEBUG: every gather index and output row is
checked against the bounds the host passed; a failed check records BAD_INDEX
and skips the access instead of touching memory out of range).

The canary cases run through the debug library: the device status must stay
OK (no check fails) and the canaries around every output stay intact; on one
ragged case its outputs must equal the release library's bit for bit.
"""

import pytest
import torch

import test_gpu_canary as canary
from helpers import ensure_built
from kv_cache_eviction_snapkv_gb300 import workloads as wk

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _use(path):
    from kv_cache_eviction_snapkv_gb300 import _native
    with _native._lock:
        _native._lib = None
        _native._LIB_PATH = path


@pytest.fixture(scope="module")
def debug_lib():
    from kv_cache_eviction_snapkv_gb300 import _native, build
    release = ensure_built()
    path = build.build(debug=True)
    _use(path)
    try:
        yield path
    finally:
        _use(release)
        assert _native.lib_path() == release


@pytest.mark.parametrize("case", canary.CASES, ids=[c[0] for c in canary.CASES])
def test_debug_library_canary_cases(debug_lib, case):
    from kv_cache_eviction_snapkv_gb300 import _native
    assert _native.lib_path() == debug_lib
    canary.test_selection_paths_stay_in_bounds(case)


def test_debug_library_other_entry_points(debug_lib):
    canary.test_grouped_and_jacap_and_reverse_stay_in_bounds()


def test_debug_library_matches_release(debug_lib):
    from kv_cache_eviction_snapkv_gb300 import api
    wl = wk.custom_workload("debug_vs_release", 2, 3, 128, 16, 300, "bf16", "avg", 5,
                            [2000, 90, 700, 300], 12)
    q, k, v = wk.device_tensors(wl, DEV)
    got = api.kvsel_snapkv(q, k, v, wl.offsets, wl.window, wl.capacity, wl.pool_kind, wl.pool_k)
    assert api.kvsel_device_status() == 0
    _use(ensure_built())
    try:
        want = api.kvsel_snapkv(q, k, v, wl.offsets, wl.window, wl.capacity, wl.pool_kind,
                                wl.pool_k)
        assert api.kvsel_device_status() == 0
    finally:
        _use(debug_lib)
    for g, w in zip(got, want):
        assert torch.equal(g, w)
