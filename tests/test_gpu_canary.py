"""Out-of-bounds write checks: every device output buffer of every entry point
sits between two 4 KiB canary regions (a fixed byte pattern), at odd shapes
(lengths that are not multiples of the 128-token tile, a one-token window, a
one-slot budget, a pooling width wider than the prefix, sequences shorter
than the budget, long prompts on the two-pass kernel). After each call the
device status must be OK and both canaries byte-for-byte untouched.
"""

import numpy as np
import pytest
import torch

from helpers import ensure_built
from kv_cache_eviction_snapkv_gb300 import workloads as wk

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
GUARD = 4096          # bytes of canary on each side
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def api():
    from kv_cache_eviction_snapkv_gb300 import api as a
    return a


class Guarded:
    """A tensor of `shape` in the middle of a buffer whose two ends hold the
    canary pattern."""

    def __init__(self, shape, dtype):
        esize = torch.empty((), dtype=dtype).element_size()
        self.g = GUARD // esize
        self.n = int(np.prod(shape))
        self.buf = torch.empty(self.n + 2 * self.g, dtype=dtype, device=DEV)
        self.buf.view(torch.uint8).fill_(PATTERN)
        self.t = self.buf[self.g:self.g + self.n].view(shape)

    def intact(self):
        b = self.buf.view(torch.uint8)
        e = b.numel() // self.buf.numel()
        head, tail = b[:self.g * e], b[(self.g + self.n) * e:]
        return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())


def check(*guarded):
    st = api().kvsel_device_status()
    assert st == 0, api().kvsel_status_string(st)
    for g in guarded:
        assert g.intact(), "a canary region was written"


CASES = [
    # name, layers, H, D, W, C, dtype, pool, k, lens
    ("w1_c2_bf16", 2, 3, 128, 1, 2, "bf16", "avg", 1, [129, 1, 300, 2, 130]),
    ("k1_pool9", 1, 2, 64, 4, 5, "bf16", "max", 9, [5, 6, 131, 4, 257]),
    ("wide_pool_f32", 1, 3, 64, 7, 9, "f32", "avg", 9, [9, 15, 100, 8]),
    ("odd_d96", 1, 2, 96, 3, 40, "bf16", "avg", 3, [333, 40, 39, 1027]),
    ("two_pass_w64", 1, 2, 128, 64, 1000, "bf16", "max", 5, [40001, 999, 64]),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_selection_paths_stay_in_bounds(case):
    name, layers, H, D, W, C, dtype, pool, kk, lens = case
    a = api()
    wl = wk.custom_workload(name, layers, H, D, W, C, dtype, pool, kk, lens, 3)
    q, k, v = wk.device_tensors(wl, DEV)
    T, t_out = wl.total, wl.out_tokens
    # fused path
    oi = Guarded((layers, t_out, H), torch.int32)
    ok_ = Guarded((layers, t_out, H, D), k.dtype)
    ov = Guarded((layers, t_out, H, D), k.dtype)
    a.kvsel_snapkv(q, k, v, wl.offsets, W, C, wl.pool_kind, kk, oi.t, ok_.t, ov.t)
    check(oi, ok_, ov)
    # stages alone
    votes = Guarded((layers, H, T), torch.float32)
    pooled = Guarded((layers, H, T), torch.float32)
    a.kvsel_score(q, k, wl.offsets, W, wl.pool_kind, kk, votes.t, pooled.t)
    check(votes, pooled)
    if T * W * layers * H <= 1 << 22:
        logits = Guarded((layers, H, W, T), torch.float32)
        a.kvsel_window_logits(q, k, wl.offsets, W, logits.t)
        check(logits)
    sel = Guarded((layers, t_out, H), torch.int32)
    a.kvsel_select(pooled.t, wl.offsets, H, W, C, sel.t)
    check(sel)
    ck = Guarded((layers, t_out, H, D), k.dtype)
    cv = Guarded((layers, t_out, H, D), k.dtype)
    a.kvsel_compact(k, v, wl.offsets, sel.t, C, ck.t, cv.t)
    check(ck, cv)
    # decode over the compacted cache, two appended rows
    kept_offs = [0] + [int(x) for x in np.cumsum([min(l, C) for l in lens])]
    qd = torch.randn((layers, len(lens), H, D), device=DEV).to(k.dtype)
    kn = torch.randn((layers, 2 * len(lens), H, D), device=DEV).to(k.dtype)
    vn = torch.randn((layers, 2 * len(lens), H, D), device=DEV).to(k.dtype)
    if a.kvsel_device_status() == 0 and D in (64, 128):
        out = Guarded((layers, len(lens), H, D), torch.float32)
        lse = Guarded((layers, len(lens), H), torch.float32)
        a.kvsel_decode_attention(qd, ok_.t, ov.t, kept_offs, kn, vn, 2, out.t, lse.t)
        check(out, lse)


def test_grouped_and_jacap_and_reverse_stay_in_bounds():
    a = api()
    # grouped selection: 4 query heads over 2 K/V heads
    wl = wk.custom_workload("canary_gqa", 1, 4, 128, 5, 70, "bf16", "avg", 3, [70, 69, 1301], 4)
    q = wk.device_tensors(wl, DEV)[0]
    wkv = wk.custom_workload("canary_gqa_kv", 1, 2, 128, 5, 70, "bf16", "avg", 3,
                             [70, 69, 1301], 5)
    _, k, v = wk.device_tensors(wkv, DEV)
    t_out = wl.out_tokens
    oi = Guarded((1, t_out, 2), torch.int32)
    ok_ = Guarded((1, t_out, 2, 128), torch.bfloat16)
    ov = Guarded((1, t_out, 2, 128), torch.bfloat16)
    a.kvsel_snapkv_grouped(q, k, v, wl.offsets, 5, 70, 0, 3, oi.t, ok_.t, ov.t)
    check(oi, ok_, ov)
    # Jacap (bf16, D = 128, H_kv = H): ragged, one short sequence
    wj = wk.custom_workload("canary_jacap", 1, 2, 128, 32, 100, "bf16", "avg", 1,
                            [1000, 90, 257], 6)
    q, k, v = wk.device_tensors(wj, DEV)
    sc = Guarded((1, 2, wj.total), torch.float32)
    a.kvsel_jacap_score(q, k, v, wj.offsets, 32, scores=sc.t)
    check(sc)
    jt = wj.out_tokens
    ji = Guarded((1, jt, 2), torch.int32)
    jk = Guarded((1, jt, 2, 128), torch.bfloat16)
    jv = Guarded((1, jt, 2, 128), torch.bfloat16)
    a.kvsel_jacap(q, k, v, wj.offsets, 32, 100, out_idx=ji.t, out_K=jk.t, out_V=jv.t)
    check(ji, jk, jv)
    # reverse-mask attention: one-row and tile-edge sequences, 4 query heads over 2
    lens = [1, 129, 300]
    n = sum(lens)
    offs = [0] + [int(x) for x in np.cumsum(lens)]
    Q = torch.randn((1, n, 4, 128), device=DEV).to(torch.bfloat16)
    K = torch.randn((1, n, 2, 128), device=DEV).to(torch.bfloat16)
    V = torch.randn((1, n, 2, 128), device=DEV).to(torch.bfloat16)
    out = Guarded((1, n, 4, 128), torch.float32)
    lse = Guarded((1, 4, n), torch.float32)
    a.kvsel_reverse_attention(Q, K, V, offs, out=out.t, lse=lse.t)
    check(out, lse)
