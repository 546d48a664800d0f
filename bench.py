#!/usr/bin/env python3
"""SnapKV selection benchmark on GB300: prompt head-tokens scored+compacted per second.

One step = one fused ``kvsel_snapkv`` call over the whole workload (score every
cached prompt token of every (layer, head), pool, select C - W, gather K/V).
Default workload: 32 layers x 32 heads (1024 instances), L = 16384, D = 128,
W = 32, C = 2048, bf16 N(0,1), avg pooling k = 7; K alone is 4 GiB per step,
far larger than L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config cfg2]
    python bench.py --impl reference ...     # the fp64 CPU oracle on host cores

Prints one JSON line (rank 0). Under torchrun each rank runs its own copy of
the workload (weak scaling, no collective on the data path); the timed region
is bracketed by barriers and the slowest rank's time is reported. At one GPU
the other named long-prompt workloads (cfg3: L = 131072, W = 64; cfg4: eight
ragged sequences; cfg5: c = 0.9) are then timed the same way, each outside
the headline's timed region, under the key "configs".
"""

from __future__ import annotations

import argparse
import dataclasses
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prompt head·tokens/s scored+compacted; achieved HBM GB/s as % of GB300 roofline"
UNIT = "head·tokens/s"


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--config", default="cfg2")
    p.add_argument("--e2e-steps", type=int, default=4)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-decode", action="store_true",
                   help="skip the decode-consumer measurement")
    p.add_argument("--no-jacap", action="store_true", help="skip the Jacap measurement")
    p.add_argument("--split", action="store_true",
                   help="with several GPUs, split the workload's layers over the ranks "
                        "(strong scaling) instead of one replica per rank (weak scaling)")
    p.add_argument("--no-gqa", action="store_true",
                   help="skip the grouped-query (group-shared selection) measurement")
    p.add_argument("--no-reverse", action="store_true",
                   help="skip the reverse-mask attention measurement")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-configs", action="store_true",
                   help="skip timing the other named workloads after the headline")
    p.add_argument("--cpu-steps", type=int, default=40)
    p.add_argument("--layers", type=int, default=0,
                   help="override the workload's layer count (small profiling cases)")
    p.add_argument("--heads", type=int, default=0,
                   help="override the workload's head count (small profiling cases)")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def describe(wl, split: bool = False) -> dict:
    return {
        "workload": f"{wl.name}: {wl.note}",
        "layers": wl.layers, "heads": wl.heads, "instances": wl.layers * wl.heads * wl.num_seqs,
        "seq_lens": wl.seq_lens, "head_dim": wl.dim, "window": wl.window,
        "capacity": wl.capacity, "pool": wl.pooling, "pool_k": wl.pool_k, "dtype": wl.dtype,
        "l2": "inputs larger than L2 (K alone exceeds the 129 MB L2 every step; no flush)",
        "parallelism": ("the workload's layers split over the GPUs, one contiguous share each "
                        "(strong scaling)" if split else
                        "one replica of the workload per GPU (weak scaling)"),
    }


# ---------------------------------------------------------------------------
# CPU oracle timing (the --impl reference arm and the cpu_baseline leg)
# ---------------------------------------------------------------------------

_HEAD = {}


def _oracle_worker(task):
    """Runs in a spawned single-threaded worker: time the oracle on one head."""
    name, layer, seq, head = task
    from kv_cache_eviction_snapkv_gb300 import workloads as wk
    import oracle
    key = (name, layer, seq, head)
    if key not in _HEAD:
        _HEAD.clear()
        wl = wk.make_workload(name)
        _HEAD[key] = (wl, wk.head_inputs(wl, layer, seq, head))
    wl, (q, k, v) = _HEAD[key]
    t0 = time.perf_counter()
    res = oracle.snapkv_head(q, k, v, wl.capacity, wl.pool_k, wl.pooling)
    dt = time.perf_counter() - t0
    return dt, len(res["indices"]), k.shape[0]


class OraclePool:
    """Single-threaded oracle processes (spawned, BLAS limited to one thread)."""

    def __init__(self, cfg: str, workers: int):
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        self.cfg = cfg
        self.workers = workers
        self.pool = mp.get_context("spawn").Pool(workers)
        from kv_cache_eviction_snapkv_gb300 import workloads as wk
        wl = wk.make_workload(cfg)
        seq = max(range(wl.num_seqs), key=lambda b: wl.seq_lens[b])
        self.task = (cfg, 0, seq, 0)
        self.tokens = wl.seq_lens[seq]
        self.pool.map(_oracle_worker, [self.task] * workers, chunksize=1)   # warm caches

    def step(self) -> float:
        t0 = time.perf_counter()
        self.pool.map(_oracle_worker, [self.task] * self.workers, chunksize=1)
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()

    def sample_text(self) -> str:
        return (f"{self.cfg}: one (layer 0, head 0) instance, L={self.tokens}, run by the fp64 "
                f"numpy oracle in each of {self.workers} single-threaded spawned processes per "
                f"step (value = {self.workers} x L head-tokens / step wall time)")


def n_workers() -> int:
    """Every host core this process may run on (one oracle process per core)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or "unknown"."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_fields(pool) -> dict:
    return {"cores": pool.workers, "host_cores": os.cpu_count(), "cpu_model": cpu_model()}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from kv_cache_eviction_snapkv_gb300 import workloads as wk
    wl = wk.make_workload(args.config)
    pool = OraclePool(args.config, n_workers())
    for _ in range(args.warmup):
        pool.step()
    times = [pool.step() for _ in range(args.steps)]
    pool.close()
    total = sum(times)
    value = pool.workers * pool.tokens * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": describe(wl),
        "cpu_baseline": {"value": value, "unit": UNIT, **cpu_fields(pool), "kind": "oracle",
                         "sample": pool.sample_text()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str):
        self.path = tempfile.mktemp(prefix="kvsel_clocks_", suffix=".csv")
        self.f = open(self.path, "w")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", uuid, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        loaded = [r for r in rows if r[2] >= 50] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in loaded for n, v in zip(names, r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in loaded), "reasons": reasons,
                "samples": len(loaded)}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def score_traffic(layers_full: int):
    """DRAM bytes per full launch of the scoring kernel from the committed ncu
    summary, scaled from the captured layer count; None when the kernel source
    (score_tc.cu and tc_common.cuh) changed since the capture (their sha256 is
    recorded beside the counters)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "score_tc_cfg2_ncu.md")
    csrc = os.path.join(ROOT, "kv_cache_eviction_snapkv_gb300", "csrc")
    try:
        text = open(path).read()
        h = hashlib.sha256()
        for name in ("score_tc.cu", "tc_common.cuh"):      # the kernel and its helpers
            h.update(open(os.path.join(csrc, name), "rb").read())
        digest = h.hexdigest()
    except OSError:
        return None
    fields = dict(line.split(":", 1) for line in text.splitlines()
                  if line.startswith(("source_sha256:", "dram_bytes_per_launch:",
                                      "captured_layers:")))
    if fields.get("source_sha256", "").strip() != digest:
        return None
    per_capture = float(fields["dram_bytes_per_launch"])
    return per_capture * layers_full / float(fields["captured_layers"])


def measure_decode(api, wl, q_win, k, v, out_k, out_v, dev, peak, peak_kind, iters=20):
    """Time kvsel_decode_attention on the compacted and the full cache (CUDA
    events on the launching stream, inputs larger than L2) and report the
    retained mass and relative output error of the compacted cache."""
    import torch
    gen = torch.Generator().manual_seed(4242)
    q = torch.randn((wl.layers, wl.num_seqs, wl.heads, wl.dim), generator=gen).to(k.dtype).to(dev)
    kept = [min(l, wl.capacity) for l in wl.seq_lens]
    kept_offs = [0] + [int(x) for x in np.cumsum(kept)]
    eb = k.element_size()
    n = wl.layers * wl.num_seqs * wl.heads
    o_keep = torch.empty((wl.layers, wl.num_seqs, wl.heads, wl.dim), dtype=torch.float32,
                         device=dev)
    o_full = torch.empty_like(o_keep)
    l_keep = torch.empty((wl.layers, wl.num_seqs, wl.heads), dtype=torch.float32, device=dev)
    l_full = torch.empty_like(l_keep)
    io = n * wl.dim * (eb + 4)          # the query in, the output out

    def timed(fn):
        for _ in range(3):
            fn()
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(iters):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / iters

    ms_keep = timed(lambda: api.kvsel_decode_attention(q, out_k, out_v, kept_offs, out=o_keep,
                                                       lse=l_keep))
    ms_full = timed(lambda: api.kvsel_decode_attention(q, k, v, wl.offsets, out=o_full,
                                                       lse=l_full))

    def quality(qq):
        api.kvsel_decode_attention(qq, out_k, out_v, kept_offs, out=o_keep, lse=l_keep)
        api.kvsel_decode_attention(qq, k, v, wl.offsets, out=o_full, lse=l_full)
        mass, err = api.kvsel_decode_quality(l_keep, l_full, o_keep, o_full)
        m = mass.flatten().double().cpu().numpy()
        return {"retained_mass": {"mean": float(m.mean()), "min": float(m.min()),
                                  "p10": float(np.percentile(m, 10))},
                "output_error": {"mean": float(err.mean()),
                                 "full_output_norm_mean": float(o_full.norm(dim=-1).mean())}}

    # a query like the window's: the last window query of each (layer, sequence, head)
    last = torch.arange(wl.num_seqs, device=dev) * wl.window + wl.window - 1
    q_last = q_win[:, last].contiguous()
    q_random = quality(q)
    q_window = quality(q_last)
    st = api.kvsel_device_status()
    if st != 0:
        raise RuntimeError(f"device status after decode: {api.kvsel_status_string(st)}")

    def line(ms, rows):
        b = wl.layers * wl.heads * rows * wl.dim * eb * 2 + io
        gbs = b / (ms * 1e-3) / 1e9
        return {"ms": ms, "bytes": b, "achieved_gbs": gbs, "frac": gbs / peak}

    return {"kernels": "decode_partial_kernel + decode_combine_kernel (2 launches per call)",
            "timed_query": "one N(0,1) query per (layer, sequence, head), g = 0",
            "compacted": line(ms_keep, sum(kept)), "full": line(ms_full, wl.total),
            "peak": peak, "peak_source": peak_kind, "unit": "GB/s",
            "quality_random_query": q_random,
            "quality_last_window_query": q_window,
            "kept_fraction": sum(kept) / wl.total}


def measure_jacap(api, wl, q_win, k, v, dev, peak, peak_kind, iters=10):
    """Time kvsel_jacap_score (statistics, Gram, factor and leverage kernels) and
    the fused kvsel_jacap (plus the selection and gather) with CUDA events."""
    import torch
    tau, beta, eps = 10.0, 0.9, 1e-6
    scores = torch.empty((wl.layers, wl.heads, wl.total), dtype=torch.float32, device=dev)
    kept = wl.out_tokens
    oi = torch.empty((wl.layers, kept, wl.heads), dtype=torch.int32, device=dev)
    ok_ = torch.empty((wl.layers, kept, wl.heads, wl.dim), dtype=k.dtype, device=dev)
    ov_ = torch.empty_like(ok_)

    def timed(fn):
        for _ in range(2):
            fn()
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(iters):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / iters

    ms_score = timed(lambda: api.kvsel_jacap_score(q_win, k, v, wl.offsets, wl.window, tau,
                                                   beta, eps, scores=scores))
    ms_full = timed(lambda: api.kvsel_jacap(q_win, k, v, wl.offsets, wl.window, wl.capacity,
                                            tau, beta, eps, oi, ok_, ov_))
    st = api.kvsel_device_status()
    if st != 0:
        raise RuntimeError(f"device status after jacap: {api.kvsel_status_string(st)}")
    eb = k.element_size()
    prefix = sum(max(0, l - wl.window) for l in wl.seq_lens)
    # K read once (statistics), V twice (Gram, leverage), the scores written
    b = wl.layers * wl.heads * prefix * (3 * wl.dim * eb + 4)
    flops = wl.layers * wl.heads * prefix * (2 * wl.dim * wl.dim) * 3   # Gram + 2 leverage MMAs
    gbs = b / (ms_score * 1e-3) / 1e9
    return {"kernels": "jacap_stats, jacap_gram (tcgen05), jacap_factor, jacap_leverage "
                       "(tcgen05)", "tau": tau, "beta": beta, "eps": eps,
            "score_ms": ms_score, "bytes": b, "achieved_gbs": gbs, "frac": gbs / peak,
            "peak": peak, "peak_source": peak_kind, "tensor_tflops": flops / (ms_score * 1e-3) / 1e12,
            "fused_ms": ms_full, "fused_head_tokens_per_s": wl.head_tokens() / (ms_full * 1e-3)}


def measure_gqa(api, wk, dev, peak, peak_kind, iters=20):
    """Group-shared selection with grouped-query attention: 4 layers, 32 query
    heads over 8 K/V heads, L = 16384, D = 128, W = 16, C = 2048, bf16 N(0,1),
    average pooling 7 (inputs larger than L2). kvsel_snapkv_grouped scores the
    four query heads of a K/V head in one MMA (64 window rows), reading K once
    per K/V head; kvsel_snapkv on the same inputs selects per query head and
    reads each K row once per query head. CUDA events on the launching stream."""
    import torch
    lens = [16384]
    wq = wk.custom_workload("gqa_q", 4, 32, 128, 16, 2048, "bf16", "avg", 7, lens, 2101)
    wkv = wk.custom_workload("gqa_kv", 4, 8, 128, 16, 2048, "bf16", "avg", 7, lens, 2102)
    q, _, _ = wk.device_tensors(wq, dev)
    _, k, v = wk.device_tensors(wkv, dev)

    def timed(fn):
        for _ in range(3):
            fn()
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(iters):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / iters
        api.kvsel_profile_begin(iters)
        for _ in range(iters):
            fn()
        stage_ms, calls = api.kvsel_profile_end()
        return ms, stage_ms[0] / calls, stage_ms[1] / calls

    offs = wq.offsets
    ms_g, score_g, sel_g = timed(lambda: api.kvsel_snapkv_grouped(q, k, v, offs, 16, 2048, 0, 7))
    ms_e, score_e, sel_e = timed(lambda: api.kvsel_snapkv(q, k, v, offs, 16, 2048, 0, 7))
    st = api.kvsel_device_status()
    if st != 0:
        raise RuntimeError(f"device status after GQA: {api.kvsel_status_string(st)}")
    row = 128 * 2
    L, layers, hq, hkv = 16384, 4, 32, 8
    qbytes = layers * hq * 16 * row
    # group-shared: K once per K/V head, the kept K/V rows of each K/V head read and written
    k_bytes = layers * hkv * L * row
    b_g = k_bytes + qbytes + layers * hkv * 4 * 2048 * row
    del q, k, v
    torch.cuda.empty_cache()
    return {"workload": "4 layers, 32 query heads over 8 K/V heads, L = 16384, D = 128, W = 16, "
                        "C = 2048, bf16 N(0,1), avg pooling 7",
            "grouped": {"entry": "kvsel_snapkv_grouped (one MMA per K tile for the 4 query "
                                 "heads of a group)",
                        "ms": ms_g, "score_ms": score_g, "select_gather_ms": sel_g,
                        "bytes": b_g, "achieved_gbs": b_g / (ms_g * 1e-3) / 1e9,
                        "frac": b_g / (ms_g * 1e-3) / 1e9 / peak,
                        "score_gbs": (k_bytes + qbytes) / (score_g * 1e-3) / 1e9,
                        "score_frac": (k_bytes + qbytes) / (score_g * 1e-3) / 1e9 / peak},
            "per_query_head": {"entry": "kvsel_snapkv (K read once per query head)",
                               "ms": ms_e, "score_ms": score_e, "select_gather_ms": sel_e},
            "peak": peak, "peak_source": peak_kind, "unit": "GB/s"}


def measure_reverse(api, dev, iters=10):
    """Reverse-mask attention of the counter-causal scorer on the shape the
    page times (one sequence of n cached rows, 28 query heads over 4 K/V heads,
    D = 128, bf16): one layer (the single-layer approximation) at n = 512 and
    n = 4096, and 28 layers at n = 4096 (the attention of the full reverse
    pass). Useful flops: QK^T and PV over the allowed pairs, 4 D n (n - 1) / 2
    per head; peak: the measured bf16 GEMM burst rate."""
    import torch
    from kv_cache_eviction_snapkv_gb300 import workloads as wk
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak_tf, peak_kind = float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        peak_tf, peak_kind = 1900.0, "fallback"
    res = {"kernel": "reverse_kernel (tcgen05, two passes, P as bf16 hi + lo)",
           "heads": 28, "kv_heads": 4, "dim": 128, "peak_tflops": peak_tf, "peak_source": peak_kind,
           "runs": []}
    for layers, n, it in ((1, 512, 4 * iters), (1, 4096, iters), (28, 4096, max(2, iters // 4))):
        q, k, v = wk.reverse_tensors(layers, n, 28, 4, 128, 2000 + n, dev)
        out = torch.empty((layers, n, 28, 128), dtype=torch.float32, device=dev)
        lse = torch.empty((layers, 28, n), dtype=torch.float32, device=dev)
        for _ in range(2):
            api.kvsel_reverse_attention(q, k, v, [0, n], out=out, lse=lse)
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(it):
            api.kvsel_reverse_attention(q, k, v, [0, n], out=out, lse=lse)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / it
        st = api.kvsel_device_status()
        if st != 0:
            raise RuntimeError(f"device status after reverse attention: {api.kvsel_status_string(st)}")
        tf = layers * 28 * 4 * 128 * n * (n - 1) / 2 / (ms * 1e-3) / 1e12
        res["runs"].append({"layers": layers, "n": n, "ms": ms, "useful_tflops": tf,
                            "frac": tf / peak_tf})
        del q, k, v, out, lse
    return res


SCORE_KERNELS = {
    1: "tc_score_kernel (window logits, softmax statistics, votes)",
    3: "tc_score_rc_kernel (statistics, then votes from logits recomputed from K in L2)",
}


def score_bytes_of(wl) -> int:
    """Algorithmic bytes of the scoring stage: K and the window queries of
    every scored (layer, sequence, head), read once."""
    eb = 2 if wl.dtype == "bf16" else 4
    scored = [l for l in wl.seq_lens if l >= wl.capacity]
    return wl.layers * wl.heads * sum((l + wl.window) * wl.dim * eb for l in scored)


def time_decode_compacted(api, wl, out_k, out_v, dev, peak, iters=20):
    """kvsel_decode_attention over a step's compacted cache (g = 0, one N(0,1)
    query per instance): CUDA events around each call, L2 flushed (256 MiB
    written) before each, since these caches can fit in L2."""
    import torch
    gen = torch.Generator().manual_seed(4243)
    q = torch.randn((wl.layers, wl.num_seqs, wl.heads, wl.dim), generator=gen).to(out_k.dtype).to(dev)
    kept = [min(l, wl.capacity) for l in wl.seq_lens]
    offs = [0] + [int(x) for x in np.cumsum(kept)]
    o = torch.empty((wl.layers, wl.num_seqs, wl.heads, wl.dim), dtype=torch.float32, device=dev)
    lse = torch.empty((wl.layers, wl.num_seqs, wl.heads), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        api.kvsel_decode_attention(q, out_k, out_v, offs, out=o, lse=lse)
    total = 0.0
    for _ in range(iters):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        api.kvsel_decode_attention(q, out_k, out_v, offs, out=o, lse=lse)
        e1.record(stream)
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1)
    ms = total / iters
    eb = out_k.element_size()
    n = wl.layers * wl.num_seqs * wl.heads
    b = wl.layers * wl.heads * sum(kept) * wl.dim * eb * 2 + n * wl.dim * (eb + 4)
    gbs = b / (ms * 1e-3) / 1e9
    del flush
    return {"ms": ms, "bytes": b, "achieved_gbs": gbs, "frac": gbs / peak,
            "l2": "flushed before each call (256 MiB written)"}


def measure_config(api, wk, name, dev, uuid, peak, steps=50, warmup=5):
    """One named workload timed like the headline step (fused kvsel_snapkv on
    device-resident inputs, CUDA events on the launching stream, clocks sampled
    during the timed region), then its stage times from the library's events."""
    import torch
    wl = wk.make_workload(name)
    q, k, v = wk.device_tensors(wl, dev)
    shape = api.shape_of(k, wl.offsets)
    t_out = api.kvsel_out_tokens(shape, wl.capacity)
    out_idx = torch.empty((wl.layers, t_out, wl.heads), dtype=torch.int32, device=dev)
    out_k = torch.empty((wl.layers, t_out, wl.heads, wl.dim), dtype=k.dtype, device=dev)
    out_v = torch.empty_like(out_k)

    def step():
        api.kvsel_snapkv(q, k, v, wl.offsets, wl.window, wl.capacity, wl.pool_kind, wl.pool_k,
                         out_idx, out_k, out_v)

    sampler = ClockSampler(uuid)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    api.kvsel_profile_begin(steps)
    for _ in range(steps):
        step()
    stage_ms, calls = api.kvsel_profile_end()
    clocks = sampler.stop()
    st = api.kvsel_device_status()
    if st != 0:
        raise RuntimeError(f"device status after {name}: {api.kvsel_status_string(st)}")
    score_ms = stage_ms[0] / calls
    step_bytes = wl.roofline_bytes()
    res = {"workload": f"{wl.name}: {wl.note}", "steps": steps, "warmup": warmup,
           "ms_per_step": ms, "value": wl.head_tokens() / (ms * 1e-3), "unit": UNIT,
           "score_kernel": SCORE_KERNELS.get(api.kvsel_score_path(shape, wl.window,
                                                                   wl.capacity), "generic"),
           "step_bytes": step_bytes,
           "step_roofline_frac": step_bytes / (ms * 1e-3) / 1e9 / peak,
           "score_bytes": score_bytes_of(wl),
           "score_frac": score_bytes_of(wl) / (score_ms * 1e-3) / 1e9 / peak,
           "stages_ms": {"score": score_ms, "select_gather": stage_ms[1] / calls,
                         "calls": calls},
           "clocks": clocks}
    res["decode_compacted"] = time_decode_compacted(api, wl, out_k, out_v, dev, peak)
    del q, k, v, out_idx, out_k, out_v
    torch.cuda.empty_cache()
    return res


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    import torch.distributed as dist

    import __graft_entry__
    from kv_cache_eviction_snapkv_gb300 import api, workloads as wk

    # Start the oracle pool (spawned) before the first GPU call.
    cpu_pool = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu_pool = OraclePool(args.config, n_workers())

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", device_id=dev)
    __graft_entry__.build()

    from kv_cache_eviction_snapkv_gb300 import shard
    wl = wk.make_workload(args.config)
    if args.layers:
        wl.layers = args.layers
    if args.heads:
        wl.heads = args.heads
    split = args.split and world > 1
    wl_full = wl
    if split:
        # strong scaling: rank r takes a contiguous share of the layers of the
        # one workload (the same bits as those layers of the whole tensors)
        share = shard.shard_range(wl.layers, rank, world)
        if len(share) == 0:
            raise SystemExit("--split needs at least one layer per rank")
        wl = dataclasses.replace(wl, layers=len(share))
        q, k, v = wk.device_tensors(wl_full, dev, layers=share)
    else:
        wl.seed = shard.rank_seed(wl.seed, rank)   # rank r's own batch (weak scaling)
        q, k, v = wk.device_tensors(wl, dev)
    shape = api.shape_of(k, wl.offsets)
    t_out = api.kvsel_out_tokens(shape, wl.capacity)
    out_idx = torch.empty((wl.layers, t_out, wl.heads), dtype=torch.int32, device=dev)
    out_k = torch.empty((wl.layers, t_out, wl.heads, wl.dim), dtype=k.dtype, device=dev)
    out_v = torch.empty_like(out_k)
    path = api.kvsel_score_path(shape, wl.window, wl.capacity)

    def step():
        api.kvsel_snapkv(q, k, v, wl.offsets, wl.window, wl.capacity, wl.pool_kind, wl.pool_k,
                         out_idx, out_k, out_v)

    def barrier():
        if world > 1:
            dist.barrier()

    uuid = str(torch.cuda.get_device_properties(dev).uuid)
    uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    sampler = ClockSampler(uuid)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = api.kvsel_device_status()
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {api.kvsel_status_string(st)}")

    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = shard.max_over_ranks(ev0.elapsed_time(ev1) / args.steps, dev)

    # Stage durations (events recorded by the library on this stream).
    n_prof = max(3, min(args.steps, 100))
    api.kvsel_profile_begin(n_prof)
    for _ in range(n_prof):
        step()
    stage_ms, calls = api.kvsel_profile_end()
    clocks = sampler.stop()
    st = api.kvsel_device_status()
    if st != 0:
        raise RuntimeError(f"device status after timing: {api.kvsel_status_string(st)}")

    score_bytes = score_bytes_of(wl)
    score_ms = stage_ms[0] / calls
    peak, peak_kind = measured_peak_gbs()
    achieved = score_bytes / (score_ms * 1e-3) / 1e9
    step_bytes = wl.roofline_bytes()
    # units of the whole job: every rank's replica (weak) or the one split workload (strong)
    units = wl.head_tokens()
    job_units = wl_full.head_tokens() if split else world * units
    job_bytes = wl_full.roofline_bytes() if split else world * step_bytes
    value = job_units / (ms * 1e-3)

    # Decode-side consumer: one N(0,1) query per (layer, sequence, head) over the
    # compacted cache this step produced and over the full prompt cache.
    decode = None
    if not args.no_decode:
        decode = measure_decode(api, wl, q, k, v, out_k, out_v, dev, peak, peak_kind)

    # Jacap scorer on the same inputs (bf16, D = 128 only).
    jacap = None
    if not args.no_jacap and wl.dtype == "bf16" and wl.dim == 128:
        jacap = measure_jacap(api, wl, q, k, v, dev, peak, peak_kind)

    # Grouped-query attention, group-shared selection (its own inputs).
    gqa = None
    if not args.no_gqa and rank == 0:
        gqa = measure_gqa(api, wk, dev, peak, peak_kind)

    # Reverse-mask attention of the counter-causal scorer (its own inputs).
    reverse = None
    if not args.no_reverse and rank == 0:
        reverse = measure_reverse(api, dev)

    # End to end through the C ABI with host buffers: kvsel_snapkv_host copies
    # q_win and K to the device layer by layer and reads the kept V rows and
    # writes the outputs in place in pinned host memory.
    e2e = None
    if not args.no_e2e:
        qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
        oih = torch.empty(out_idx.shape, dtype=out_idx.dtype, pin_memory=True)
        okh = torch.empty(out_k.shape, dtype=out_k.dtype, pin_memory=True)
        ovh = torch.empty(out_v.shape, dtype=out_v.dtype, pin_memory=True)

        def e2e_step():
            api.kvsel_snapkv_host(qh, kh, vh, wl.offsets, wl.window, wl.capacity, wl.pool_kind,
                                  wl.pool_k, oih, okh, ovh)

        for _ in range(2):
            e2e_step()
        barrier()
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier()
        st = api.kvsel_device_status()
        if st != 0:
            raise RuntimeError(f"device status after e2e: {api.kvsel_status_string(st)}")
        e2e_ms = shard.max_over_ranks(ev0.elapsed_time(ev1) / args.e2e_steps, dev)
        nbytes = lambda t: t.numel() * t.element_size()
        kept_v = out_v.numel() * out_v.element_size()   # the V rows the gather reads
        e2e = {"value": job_units / (e2e_ms * 1e-3), "unit": UNIT,
               "ms_per_step": e2e_ms, "steps": args.e2e_steps,
               "h2d_bytes_per_step": nbytes(q) + nbytes(k) + kept_v,
               "d2h_bytes_per_step": nbytes(out_idx) + nbytes(out_k) + nbytes(out_v),
               "path": "kvsel_snapkv_host: q_win and K copied per layer (two device slots, "
                       "copy stream), kept V rows read and outputs written in place in "
                       "pinned host memory"}
        del qh, kh, vh, oih, okh, ovh

    cpu = None
    if cpu_pool is not None:
        times = [cpu_pool.step() for _ in range(args.cpu_steps)]
        cpu_pool.close()
        cpu_val = cpu_pool.workers * cpu_pool.tokens * len(times) / sum(times)
        cpu = {"value": cpu_val, "unit": UNIT, **cpu_fields(cpu_pool), "kind": "oracle",
               "sample": cpu_pool.sample_text()}

    # The other long-prompt workloads, each timed like the headline step
    # (outside the headline's timed region; one GPU only).
    configs = None
    if rank == 0 and world == 1 and not args.no_configs:
        del q, k, v, out_k, out_v
        torch.cuda.empty_cache()
        configs = {}
        for name in ("cfg2", "cfg3", "cfg4", "cfg5"):
            if name != args.config:
                configs[name] = measure_config(api, wk, name, dev, uuid, peak)

    if rank == 0:
        # score kernel(s) + select/gather: one tensor-core pass, two (row split),
        # or the CUDA-core statistics, merge and votes kernels
        launches_per_step = {1: 2, 3: 2}.get(path, 4)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "strong" if split else "weak",
            "vs_baseline": None,
            "dtype": wl.dtype, "data": "synthetic (seeded counter-based generator)",
            "config": describe(wl_full, split),
            "gbs": job_bytes / (ms * 1e-3) / 1e9,
            "step_roofline_frac": step_bytes / (ms * 1e-3) / 1e9 / peak,
            "roofline": {"bound": "hbm", "kernel": SCORE_KERNELS.get(path,
                                                                     "generic scoring kernels"),
                         "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind,
                         "traffic": score_traffic(wl.layers) if path == 1 and
                         args.config == "cfg2" else None,
                         "bytes_per_launch": score_bytes,
                         "avg_launch_ms": score_ms},
            "stages_ms": {"score": stage_ms[0] / calls, "select_gather": stage_ms[1] / calls,
                          "calls": calls},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "decode": decode,
            "jacap": jacap,
            "reverse": reverse,
            "gqa": gqa,
            "configs": configs,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
