"""Seeded input generator: numpy and torch routes give the same bits, per-head
regeneration matches the whole tensor, and the planted / duplicated structure
is what the workload descriptions promise."""

import math

import numpy as np
import pytest
import torch

from kv_cache_eviction_snapkv_gb300 import workloads as wk


def test_splitmix_reference_values():
    # SplitMix64 seeded with 0: first outputs of the published generator.
    assert wk._mix_int(0 + wk.GAMMA) == 0xE220A8397B1DCDAF
    assert wk._mix_int(2 * wk.GAMMA) == 0x6E789E6AA1B965F4


def test_codes_numpy_equals_torch():
    s = wk.stream_seed(123, wk.KIND_K)
    e = np.arange(4096, dtype=np.int64)
    assert np.array_equal(wk.codes_np(s, e), wk.codes_torch(s, 0, 4096, "cpu").numpy())
    assert np.array_equal(wk.codes_np(s, e + 8192), wk.codes_torch(s, 8192, 4096, "cpu").numpy())


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_host_equals_torch_route(dtype):
    wl = wk.custom_workload("t", 2, 3, 16, 4, 24, dtype, "avg", 3, [40, 17, 64], 99,
                            plant=4, dup_fraction=0.25)
    hq, hk, hv = wk.host_tensors(wl)
    dq, dk, dv = wk.device_tensors(wl, "cpu", chunk=1 << 10)
    for h, d in ((hq, dq), (hk, dk), (hv, dv)):
        ht = wk.storage_to_torch(h, dtype)
        assert torch.equal(ht.view(torch.int16) if dtype == "bf16" else ht,
                           d.view(torch.int16) if dtype == "bf16" else d)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_layer_ranges_match_the_whole_tensors(dtype):
    """A rank's share of a workload split by layers has the same bits as the
    matching slices of the whole tensors (odd element counts per layer, so the
    shares start inside a group of four generated codes)."""
    wl = wk.custom_workload("s", 5, 3, 6, 3, 20, dtype, "avg", 3, [41, 17, 30], 77,
                            plant=3, dup_fraction=0.25)
    whole = wk.device_tensors(wl, "cpu", chunk=1 << 8)
    for rng in (range(0, 2), range(2, 5), range(1, 2), range(4, 5)):
        part = wk.device_tensors(wl, "cpu", chunk=1 << 8, layers=rng)
        for w, p in zip(whole, part):
            a = w[rng.start:rng.stop]
            assert p.shape == a.shape
            assert torch.equal(a.view(torch.int16) if dtype == "bf16" else a,
                               p.view(torch.int16) if dtype == "bf16" else p)
    with pytest.raises(ValueError):
        wk.device_tensors(wl, "cpu", layers=range(3, 6))


def test_planted_logits_rise_by_six():
    wl = wk.custom_workload("p", 1, 2, 128, 8, 64, "bf16", "max", 5, [300], 5, plant=8)
    for h in range(2):
        q, k, _ = wk.head_inputs(wl, 0, 0, h)
        pos, _ = wk._plant_rows(wl, 0, 0, h)
        plain = wk.storage_to_f64(
            wk._draw(wl, wk.KIND_K, wl.total, 0, np.array(pos), h), "bf16")
        rise = ((k[pos] - plain) * q).sum(axis=1) / math.sqrt(128)
        np.testing.assert_allclose(rise, 6.0, atol=0.1)       # bf16 rounding of k


def test_duplicated_blocks_are_exact_copies():
    wl = wk.custom_workload("d", 1, 1, 32, 16, 100, "bf16", "avg", 3, [1040], 8,
                            kv_dist=("t3grid", 1.0), dup_fraction=0.25)
    _, k, _ = wk.head_inputs(wl, 0, 0, 0)
    dst, src = wk._dup_map(wl, 0, 0, 0)
    assert len(dst) == 8 * round(0.25 * (1024 // 8))
    assert np.array_equal(k[dst], k[src])
    assert np.all(src < dst)
    grid = k * 64.0
    assert np.array_equal(grid, np.round(grid))                # values on the 1/64 grid


def test_tables():
    n = wk.bf16_bits_to_f64(wk.table("normal", "bf16"))
    assert abs(n.mean()) < 1e-6 and abs(n.std() - 1.0) < 1e-3
    assert np.all(np.diff(n) >= 0)
    t = wk.bf16_bits_to_f64(wk.table("t3grid", "bf16"))
    assert np.all(np.diff(t) >= 0) and abs(np.median(t)) < 1e-9


def test_named_workloads():
    c2 = wk.make_workload("cfg2")
    assert c2.layers * c2.heads == 1024 and c2.seq_lens == [16384]
    assert c2.roofline_bytes() == 1024 * (16384 * 256 + 32 * 256 + 4 * 2048 * 256)
    c4 = wk.make_workload("cfg4")
    assert len(c4.seq_lens) == 8
    assert sum(l < c4.capacity for l in c4.seq_lens) == 1
    assert all(4096 <= l <= 32768 for l in c4.seq_lens if l >= c4.capacity)
    c5 = wk.make_workload("cfg5")
    assert c5.capacity == round(0.1 * 65536)
