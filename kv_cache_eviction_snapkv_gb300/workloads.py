"""Seeded synthetic inputs for SnapKV selection (input construction only).

This module builds the prompt Q/K/V tensors that the tests, the benchmark and
the smoke check feed to both the CUDA library and the CPU oracle. It holds
none of the selection arithmetic.

Generator: every element is an independent draw from a counter-based stream,
so any (layer, head) slice can be rebuilt on the host without building the
whole tensor:

* stream seed  s = SplitMix64 output for (seed, tensor kind);
* group g of 4 consecutive elements (row-major in the canonical layout) takes
  the g-th SplitMix64 output h = mix(s + (g + 1) * 0x9E3779B97F4A7C15) and
  splits it into four 16-bit codes (low bits first);
* a code c becomes table[c], where table[c] is the (c + 0.5) / 65536 quantile
  of the element distribution, rounded once to the storage dtype.

SplitMix64 is Steele, Lea and Flood, "Fast splittable pseudorandom number
generators" (OOPSLA 2014). The numpy and torch routes below produce the same
bits; tests check that. Canonical layouts: q_win (layers, S*W, H, D),
K and V (layers, T, H, D).
"""

from __future__ import annotations

import math
import statistics
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1
KIND_Q, KIND_K, KIND_V = 1, 2, 3


# ---------------------------------------------------------------------------
# SplitMix64, numpy (uint64) and torch (int64 two's-complement) routes
# ---------------------------------------------------------------------------

def _mix_int(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def stream_seed(seed: int, kind: int) -> int:
    return _mix_int((seed * 16 + kind) * GAMMA + GAMMA)


def _mix_np(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX2)
        return z ^ (z >> np.uint64(31))


def codes_np(s: int, elem: np.ndarray) -> np.ndarray:
    """16-bit codes of the elements with linear indices ``elem`` (int64 array)."""
    elem = np.asarray(elem, dtype=np.uint64)
    g = elem >> np.uint64(2)
    with np.errstate(over="ignore"):
        h = _mix_np(np.uint64(s) + (g + np.uint64(1)) * np.uint64(GAMMA))
    shift = (elem & np.uint64(3)) * np.uint64(16)
    return ((h >> shift) & np.uint64(0xFFFF)).astype(np.int64)


def _signed(x: int) -> int:
    return x - (1 << 64) if x >= (1 << 63) else x


def _lsr_t(z, s: int):
    return (z >> s) & ((1 << (64 - s)) - 1)


def codes_torch(s: int, first: int, count: int, device):
    """Codes of elements first .. first+count-1 (count a multiple of 4) as int64."""
    import torch
    assert first % 4 == 0 and count % 4 == 0
    g = torch.arange(first // 4, (first + count) // 4, dtype=torch.int64, device=device)
    z = (g + 1) * _signed(GAMMA) + _signed(s)
    z = (z ^ _lsr_t(z, 30)) * _signed(MIX1)
    z = (z ^ _lsr_t(z, 27)) * _signed(MIX2)
    z = z ^ _lsr_t(z, 31)
    parts = [z & 0xFFFF] + [(_lsr_t(z, 16 * i) & 0xFFFF) for i in range(1, 4)]
    return torch.stack(parts, dim=1).reshape(-1)


# ---------------------------------------------------------------------------
# Quantile tables
# ---------------------------------------------------------------------------

def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round to fp32, then to bf16 with round-to-nearest-even; returns uint16 bits."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _uniform_midpoints() -> np.ndarray:
    return (np.arange(65536, dtype=np.float64) + 0.5) / 65536.0


def _normal_quantiles() -> np.ndarray:
    nd = statistics.NormalDist()
    return np.array([nd.inv_cdf(u) for u in _uniform_midpoints()])


def _t3_quantiles() -> np.ndarray:
    """Student-t (3 dof) quantiles by bisection on its closed-form CDF
    F(t) = 1/2 + (t / (sqrt(3) (1 + t^2/3)) + atan(t / sqrt(3))) / pi."""
    u = _uniform_midpoints()
    lo, hi = np.full(u.shape, -1e3), np.full(u.shape, 1e3)
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        x = mid / math.sqrt(3.0)
        cdf = 0.5 + (x / (1.0 + x * x) + np.arctan(x)) / math.pi
        below = cdf < u
        lo = np.where(below, mid, lo)
        hi = np.where(below, hi, mid)
    return 0.5 * (lo + hi)


_TABLES: Dict[Tuple[str, str, float], np.ndarray] = {}


def table(dist: str, dtype: str, scale: float = 1.0) -> np.ndarray:
    """Storage-format table: uint16 bf16 bits or float32 values, 65536 entries.

    dist: "normal" (N(0,1) * scale) or "t3grid" (0.5 * t3 rounded to a
    multiple of 1/64).
    """
    key = (dist, dtype, float(scale))
    if key not in _TABLES:
        if dist == "normal":
            v = _normal_quantiles() * scale
        elif dist == "t3grid":
            v = np.round(0.5 * _t3_quantiles() * 64.0) / 64.0
        else:
            raise ValueError(dist)
        _TABLES[key] = f64_to_bf16_bits(v) if dtype == "bf16" else v.astype(np.float32)
    return _TABLES[key]


def storage_to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_to_f64(x) if dtype == "bf16" else np.asarray(x, np.float64)


# ---------------------------------------------------------------------------
# Workload descriptions
# ---------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    layers: int
    heads: int
    dim: int
    window: int
    capacity: int
    dtype: str                     # "bf16" or "f32"
    pooling: str                   # "avg" or "max"
    pool_k: int
    seq_lens: List[int]
    seed: int
    q_dist: Tuple[str, float] = ("normal", 1.0)
    kv_dist: Tuple[str, float] = ("normal", 1.0)
    plant: int = 0                 # planted keys per head (logit +6 for one query)
    dup_fraction: float = 0.0      # fraction of 8-row prefix K blocks copied from earlier blocks
    note: str = ""
    _cache: Dict = field(default_factory=dict, repr=False)

    @property
    def num_seqs(self) -> int:
        return len(self.seq_lens)

    @property
    def offsets(self) -> List[int]:
        return [0] + list(np.cumsum(self.seq_lens).astype(int))

    @property
    def total(self) -> int:
        return int(sum(self.seq_lens))

    @property
    def out_tokens(self) -> int:
        return int(sum(min(l, self.capacity) for l in self.seq_lens))

    @property
    def pool_kind(self) -> int:
        return 0 if self.pooling == "avg" else 1

    def q_shape(self):
        return (self.layers, self.num_seqs * self.window, self.heads, self.dim)

    def kv_shape(self):
        return (self.layers, self.total, self.heads, self.dim)

    def head_tokens(self) -> int:
        """Prompt head-tokens (sum over layers, heads, sequences of L_b)."""
        return self.layers * self.heads * self.total

    def roofline_bytes(self) -> int:
        """Algorithmic bytes: per (layer, head, seq) L*D*eb of K + W*D*eb of q
        + 4*C*D*eb of selected K/V read and written; bypass: 4*L*D*eb."""
        eb = 2 if self.dtype == "bf16" else 4
        row = self.dim * eb
        per_head = 0
        for l in self.seq_lens:
            if l < self.capacity:
                per_head += 4 * l * row
            else:
                per_head += l * row + self.window * row + 4 * self.capacity * row
        return self.layers * self.heads * per_head


def make_workload(name: str) -> Workload:
    """The named synthetic configurations (seeds are 1000 + config number)."""
    if name == "cfg1":
        return Workload("cfg1", 1, 4, 64, 32, 256, "f32", "avg", 7, [1024], 1001,
                        q_dist=("normal", 2.0 / 8.0), kv_dist=("normal", 2.0 / 8.0),
                        note="MHA 4 heads, L=1024, D=64, fp32, N(0,1)*2/sqrt(D)")
    if name == "cfg2":
        return Workload("cfg2", 32, 32, 128, 32, 2048, "bf16", "avg", 7, [16384], 1002,
                        note="32 layers x 32 heads, L=16384, D=128, bf16 N(0,1)")
    if name == "cfg3":
        return Workload("cfg3", 1, 32, 128, 64, 4096, "bf16", "max", 5, [131072], 1003,
                        plant=64, note="32 heads, L=131072, 64 planted keys (+6 logit)")
    if name == "cfg4":
        rng = np.random.default_rng(np.random.SeedSequence([1004, 0]))
        lens = [int(x) for x in rng.integers(4096, 32768, size=7, endpoint=True)]
        short = int(rng.integers(32, 1024 - 1, endpoint=True))
        pos = int(rng.integers(0, 8))
        lens.insert(pos, short)
        return Workload("cfg4", 1, 32, 128, 32, 1024, "bf16", "avg", 7, lens, 1004,
                        note="ragged 8 sequences, one shorter than C (bypass)")
    if name == "cfg5":
        return Workload("cfg5", 1, 32, 128, 16, 6554, "bf16", "avg", 3, [65536], 1005,
                        kv_dist=("t3grid", 1.0), dup_fraction=0.25,
                        note="c=0.9, keys 0.5*t(3) on a 1/64 grid, 25% duplicated 8-row blocks")
    raise KeyError(name)


def custom_workload(name, layers, heads, dim, window, capacity, dtype, pooling, pool_k,
                    seq_lens, seed, **kw) -> Workload:
    return Workload(name, layers, heads, dim, window, capacity, dtype, pooling, pool_k,
                    list(seq_lens), seed, **kw)


# ---------------------------------------------------------------------------
# Element addressing and per-head host regeneration
# ---------------------------------------------------------------------------

def _tables(wl: Workload):
    tq = table(wl.q_dist[0], wl.dtype, wl.q_dist[1])
    tkv = table(wl.kv_dist[0], wl.dtype, wl.kv_dist[1])
    return tq, tkv


def _elements(rows_total: int, wl: Workload, layer: int, rows: np.ndarray, head: int):
    """Linear element indices of (layer, rows, head, 0..D-1) in the canonical layout."""
    d = np.arange(wl.dim, dtype=np.int64)
    base = ((layer * rows_total + rows.astype(np.int64)) * wl.heads + head) * wl.dim
    return (base[:, None] + d[None, :]).reshape(-1)


def _draw(wl: Workload, kind: int, rows_total: int, layer: int, rows: np.ndarray, head: int):
    tq, tkv = _tables(wl)
    tab = tq if kind == KIND_Q else tkv
    c = codes_np(stream_seed(wl.seed, kind), _elements(rows_total, wl, layer, rows, head))
    return tab[c].reshape(len(rows), wl.dim)


def _plant_rows(wl: Workload, layer: int, seq: int, head: int):
    """(positions, new K rows in storage format) planted for one head, or None."""
    if not wl.plant:
        return None
    length = wl.seq_lens[seq]
    prefix = length - wl.window
    n = min(wl.plant, wl.window, prefix)
    rng = np.random.default_rng(np.random.SeedSequence([wl.seed, 77, layer, seq, head]))
    pos = np.sort(rng.choice(prefix, size=n, replace=False))
    qrows = np.arange(seq * wl.window, seq * wl.window + n)
    q = storage_to_f64(_draw(wl, KIND_Q, wl.num_seqs * wl.window, layer, qrows, head), wl.dtype)
    krows = wl.offsets[seq] + pos
    k = storage_to_f64(_draw(wl, KIND_K, wl.total, layer, krows, head), wl.dtype)
    # logit of window query i with planted key i rises by exactly 6 (before rounding)
    k = k + 6.0 * math.sqrt(wl.dim) * q / (q * q).sum(axis=1, keepdims=True)
    new = f64_to_bf16_bits(k) if wl.dtype == "bf16" else k.astype(np.float32)
    return pos, new


def _dup_map(wl: Workload, layer: int, seq: int, head: int):
    """(dst_rows, src_rows) within the sequence: 8-row prefix blocks copied from
    earlier blocks; chains resolved so every source is an untouched block."""
    if not wl.dup_fraction:
        return None
    length = wl.seq_lens[seq]
    prefix = length - wl.window
    nblk = prefix // 8
    if nblk < 2:
        return None
    rng = np.random.default_rng(np.random.SeedSequence([wl.seed, 88, layer, seq, head]))
    ndst = int(round(wl.dup_fraction * nblk))
    dst = np.sort(rng.choice(np.arange(1, nblk), size=min(ndst, nblk - 1), replace=False))
    root = np.arange(nblk)
    for b in dst:
        root[b] = root[int(rng.integers(0, b))]
    src = root[dst]
    off = np.arange(8)
    return ((dst[:, None] * 8 + off).reshape(-1), (src[:, None] * 8 + off).reshape(-1))


def head_inputs(wl: Workload, layer: int, seq: int, head: int, as_f64: bool = True):
    """(q_win, K, V) of one (layer, sequence, head), exactly as stored."""
    w0 = seq * wl.window
    q = _draw(wl, KIND_Q, wl.num_seqs * wl.window, layer, np.arange(w0, w0 + wl.window), head)
    o, length = wl.offsets[seq], wl.seq_lens[seq]
    rows = np.arange(o, o + length)
    k = _draw(wl, KIND_K, wl.total, layer, rows, head)
    v = _draw(wl, KIND_V, wl.total, layer, rows, head)
    dm = _dup_map(wl, layer, seq, head)
    if dm is not None:
        k[dm[0]] = k[dm[1]]
    pl = _plant_rows(wl, layer, seq, head)
    if pl is not None:
        k[pl[0]] = pl[1]
    if as_f64:
        return (storage_to_f64(q, wl.dtype), storage_to_f64(k, wl.dtype),
                storage_to_f64(v, wl.dtype))
    return q, k, v


def host_tensors(wl: Workload):
    """Whole tensors in storage format (numpy): q_win, K, V. Small workloads only."""
    sdt = np.uint16 if wl.dtype == "bf16" else np.float32
    q = np.empty(wl.q_shape(), sdt)
    k = np.empty(wl.kv_shape(), sdt)
    v = np.empty(wl.kv_shape(), sdt)
    for layer in range(wl.layers):
        for b in range(wl.num_seqs):
            o, length = wl.offsets[b], wl.seq_lens[b]
            for h in range(wl.heads):
                qh, kh, vh = head_inputs(wl, layer, b, h, as_f64=False)
                q[layer, b * wl.window:(b + 1) * wl.window, h] = qh
                k[layer, o:o + length, h] = kh
                v[layer, o:o + length, h] = vh
    return q, k, v


def device_tensors(wl: Workload, device, chunk: int = 1 << 26, layers: Optional[range] = None):
    """Whole tensors generated with torch on ``device`` (same bits as host_tensors).

    ``layers`` (a contiguous range of the workload's layers, default all): only
    those layers, with the same bits as the matching slices of the whole
    tensors (a rank's share when one workload is split over ranks)."""
    import torch
    if layers is None:
        layers = range(wl.layers)
    if layers.step != 1 or layers.start < 0 or layers.stop > wl.layers:
        raise ValueError("layers must be a contiguous range of the workload's layers")
    nl = len(layers)
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    tq, tkv = _tables(wl)

    def tab_t(t):
        if wl.dtype == "bf16":
            return torch.from_numpy(t.view(np.int16).copy()).to(device)
        return torch.from_numpy(t.copy()).to(device)

    def fill(shape, kind, tab):
        per_layer = int(np.prod(shape[1:]))
        n = nl * per_layer
        base = layers.start * per_layer        # linear index of the first element
        flat = torch.empty(n, dtype=torch.int16 if wl.dtype == "bf16" else torch.float32,
                           device=device)
        s = stream_seed(wl.seed, kind)
        lead = base % 4                         # codes come in groups of four elements
        total = lead + n + (-(lead + n)) % 4
        for first in range(0, total, chunk):
            cnt = min(chunk, total - first)
            c = codes_torch(s, base - lead + first, cnt, device)
            vals = tab[c]
            lo = max(first, lead)
            hi = min(first + cnt, lead + n)
            if hi > lo:
                flat[lo - lead:hi - lead] = vals[lo - first:hi - first]
        if wl.dtype == "bf16":
            flat = flat.view(torch.bfloat16)
        return flat.view((nl,) + tuple(shape[1:]))

    tqd, tkvd = tab_t(tq), tab_t(tkv)
    q = fill(wl.q_shape(), KIND_Q, tqd)
    k = fill(wl.kv_shape(), KIND_K, tkvd)
    v = fill(wl.kv_shape(), KIND_V, tkvd)
    for li, layer in enumerate(layers):
        for b in range(wl.num_seqs):
            o = wl.offsets[b]
            for h in range(wl.heads):
                dm = _dup_map(wl, layer, b, h)
                if dm is not None:
                    dst = torch.from_numpy(o + dm[0]).to(device)
                    src = torch.from_numpy(o + dm[1]).to(device)
                    k[li, dst, h] = k[li, src, h]
                pl = _plant_rows(wl, layer, b, h)
                if pl is not None:
                    rows = torch.from_numpy(o + pl[0]).to(device)
                    new = pl[1].view(np.int16) if wl.dtype == "bf16" else pl[1]
                    vals = torch.from_numpy(np.ascontiguousarray(new)).to(device)
                    if wl.dtype == "bf16":
                        vals = vals.view(torch.bfloat16)
                    k[li, rows, h] = vals
    return q.contiguous(), k.contiguous(), v.contiguous()


def reverse_tensors(layers: int, n: int, heads: int, kv_heads: int, dim: int, seed: int,
                    device):
    """Inputs of the reverse-mask attention: Q [layers, n, heads, dim] and K, V
    [layers, n, kv_heads, dim], bf16 N(0,1) quantiles from the counter-based
    generator (one sequence of n cached rows; Q and K/V from two streams)."""
    wq = custom_workload("reverse_q", layers, heads, dim, n, n + 1, "bf16", "avg", 1, [n], seed)
    wkv = custom_workload("reverse_kv", layers, kv_heads, dim, 1, n + 1, "bf16", "avg", 1, [n],
                          seed + 7919)
    q = device_tensors(wq, device)[0]
    _, k, v = device_tensors(wkv, device)
    return q, k, v


def storage_to_torch(x: np.ndarray, dtype: str):
    """numpy storage array -> CPU torch tensor of the storage dtype (no copy of bits)."""
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x))
