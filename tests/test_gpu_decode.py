"""Decode-side consumer on the GPU against the fp64 oracle.

One future query per (layer, sequence, head) over the compacted cache that
kvsel_snapkv produced (plus g appended rows) and over the full cache; the
retained mass and the output error from kvsel_decode_quality against the
oracle's decomposition. Bars: out within 2e-5 absolute plus 1e-4 relative, lse
within 1e-4 absolute (fp32 accumulation over the same bf16/fp32 values the
oracle reads in fp64); mass within 1e-4 absolute.
"""

import numpy as np
import pytest
import torch

import oracle
from helpers import ensure_built
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


def f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def rand(shape, gen, dtype):
    return torch.randn(shape, generator=gen).to(dtype)


def check(out, lse, ref):
    np.testing.assert_allclose(f64(out), ref["out"], rtol=1e-4, atol=2e-5)
    np.testing.assert_allclose(f64(lse), ref["lse"], rtol=0, atol=1e-4)


@pytest.mark.parametrize("dtype,D,g", [(torch.bfloat16, 128, 5), (torch.float32, 64, 0),
                                       (torch.bfloat16, 64, 513)])
def test_compacted_and_full_cache(dtype, D, g):
    """Decode over kvsel_snapkv's compacted rows and over the full prompt, with
    g appended rows; chunk boundaries (512 rows) inside and at the edges."""
    name = "dec_bf16" if dtype == torch.bfloat16 else "dec_f32"
    wl = wk.custom_workload(name, 2, 3, D, 32, 512, "bf16" if dtype == torch.bfloat16 else "f32",
                            "avg", 7, [1800, 200, 512, 513, 2600], 91)
    q_win, K, V = wk.device_tensors(wl, DEV)
    out_idx, out_k, out_v = api().kvsel_snapkv(q_win, K, V, wl.offsets, wl.window, wl.capacity,
                                               wl.pool_kind, wl.pool_k)
    assert_ok()
    gen = torch.Generator().manual_seed(5)
    S, H, L = wl.num_seqs, wl.heads, wl.layers
    q = rand((L, S, H, D), gen, dtype).to(DEV)
    kn = rand((L, S * g, H, D), gen, dtype).to(DEV) if g else None
    vn = rand((L, S * g, H, D), gen, dtype).to(DEV) if g else None
    kept_offs = [0] + list(np.cumsum([min(x, wl.capacity) for x in wl.seq_lens]))
    o_keep, l_keep = api().kvsel_decode_attention(q, out_k, out_v, kept_offs, kn, vn, g)
    o_full, l_full = api().kvsel_decode_attention(q, K, V, wl.offsets, kn, vn, g)
    assert_ok()
    kn64 = f64(kn) if g else None
    vn64 = f64(vn) if g else None
    ref_keep = oracle.decode_packed(f64(q), f64(out_k), f64(out_v), kept_offs, kn64, vn64, g)
    ref_full = oracle.decode_packed(f64(q), f64(K), f64(V), wl.offsets, kn64, vn64, g)
    check(o_keep, l_keep, ref_keep)
    check(o_full, l_full, ref_full)
    # retained mass and error, on the device, against the oracle's decomposition
    mass, err = api().kvsel_decode_quality(l_keep, l_full, o_keep, o_full)
    assert_ok()
    idx = out_idx.cpu().numpy()
    q64, k64, v64 = f64(q), f64(K), f64(V)
    for layer in range(L):
        oo = 0
        for b, length in enumerate(wl.seq_lens):
            n = min(length, wl.capacity)
            o = wl.offsets[b]
            for h in range(H):
                kr, vr = k64[layer, o:o + length, h], v64[layer, o:o + length, h]
                if g:
                    kr = np.concatenate([kr, kn64[layer, b * g:(b + 1) * g, h]])
                    vr = np.concatenate([vr, vn64[layer, b * g:(b + 1) * g, h]])
                kept = list(idx[layer, oo:oo + n, h]) + list(range(length, length + g))
                r = oracle.decompose(q64[layer, b, h], kr, vr, kept)
                assert float(mass[layer, b, h]) == pytest.approx(r["m"], abs=1e-4)
                assert float(err[layer, b, h]) == pytest.approx(r["err"], abs=5e-4)
                if length < wl.capacity and g == 0:
                    assert float(mass[layer, b, h]) == pytest.approx(1.0, abs=1e-5)
            oo += n


def test_gqa_heads_read_their_group():
    gen = torch.Generator().manual_seed(6)
    L, S, H, Hkv, D = 1, 2, 8, 2, 128
    offs = [0, 700, 1100]
    q = rand((L, S, H, D), gen, torch.bfloat16).to(DEV)
    K = rand((L, 1100, Hkv, D), gen, torch.bfloat16).to(DEV)
    V = rand((L, 1100, Hkv, D), gen, torch.bfloat16).to(DEV)
    out, lse = api().kvsel_decode_attention(q, K, V, offs)
    assert_ok()
    check(out, lse, oracle.decode_packed(f64(q), f64(K), f64(V), offs))


def test_joint_permutation_leaves_the_output():
    gen = torch.Generator().manual_seed(7)
    L, S, H, D = 1, 1, 2, 64
    q = rand((L, S, H, D), gen, torch.float32).to(DEV)
    K = rand((L, 3000, H, D), gen, torch.float32).to(DEV)
    V = rand((L, 3000, H, D), gen, torch.float32).to(DEV)
    perm = torch.randperm(3000, generator=gen).to(DEV)
    o1, l1 = api().kvsel_decode_attention(q, K, V, [0, 3000])
    o2, l2 = api().kvsel_decode_attention(q, K[:, perm].contiguous(), V[:, perm].contiguous(),
                                          [0, 3000])
    o3, _ = api().kvsel_decode_attention(q, K, V[:, perm].contiguous(), [0, 3000])
    assert_ok()
    torch.testing.assert_close(o2, o1, rtol=1e-5, atol=1e-6)
    torch.testing.assert_close(l2, l1, rtol=0, atol=1e-5)
    assert (o3 - o1).abs().max().item() > 1e-3


def test_page_example_equal_logits():
    """Two equal logits with V = [0, 10] (first dimension): full output 5, the
    first row alone 0, retained mass 1/2."""
    D = 64
    K = torch.zeros((1, 2, 1, D), device=DEV)
    K[0, :, 0, 0] = 0.25
    V = torch.zeros((1, 2, 1, D), device=DEV)
    V[0, 1, 0, 0] = 10.0
    q = torch.zeros((1, 1, 1, D), device=DEV)
    q[0, 0, 0, 0] = 1.0
    o_full, l_full = api().kvsel_decode_attention(q, K, V, [0, 2])
    o_keep, l_keep = api().kvsel_decode_attention(q, K[:, :1].contiguous(), V[:, :1].contiguous(),
                                                  [0, 1])
    mass, err = api().kvsel_decode_quality(l_keep, l_full, o_keep, o_full)
    assert_ok()
    assert o_full[0, 0, 0, 0].item() == pytest.approx(5.0, abs=1e-5)
    assert o_keep[0, 0, 0, 0].item() == 0.0
    assert mass.item() == pytest.approx(0.5, abs=1e-6)
    assert err.item() == pytest.approx(5.0, abs=1e-5)


def test_nonfinite_key_is_reported():
    q = torch.ones((1, 1, 1, 64), device=DEV)
    K = torch.zeros((1, 10, 1, 64), device=DEV)
    K[0, 3, 0, 5] = float("nan")
    V = torch.ones((1, 10, 1, 64), device=DEV)
    api().kvsel_decode_attention(q, K, V, [0, 10])
    assert api().kvsel_device_status() == api().KVSEL_ERR_NONFINITE
    assert api().kvsel_device_status() == 0
