"""bench.py's host logic on CPU: the reference arm's JSON line (the oracle
timed on the host cores), the clock record taken from nvidia-smi's CSV, the
DRAM traffic figure tied to the kernel source it was captured on, and the
workload description of both scaling modes."""

import json
import os
import shutil
import subprocess
import sys

import bench
from kv_cache_eviction_snapkv_gb300 import workloads as wk


def test_reference_arm_json_line():
    res = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl",
                          "reference", "--steps", "1", "--warmup", "1"],
                         capture_output=True, text=True, timeout=600, cwd=bench.ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["steps"] == 1 and line["warmup"] == 1 and line["n_gpus"] == 1
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"]
    assert cb["cores"] >= 1 and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": bench.UNIT,
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert line["config"]["workload"].startswith("cfg2")


def test_clock_record_from_csv(monkeypatch):
    def no_smi(*args, **kwargs):
        raise OSError("no nvidia-smi")

    monkeypatch.setattr(bench.subprocess, "Popen", no_smi)
    s = bench.ClockSampler("GPU-test")
    # sm, max sm, power, utilisation, reasons mask, hw_slowdown, hw_thermal,
    # sw_thermal, sw_power_cap
    rows = [
        "2070, 2070, 900.1, 100, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2040, 2070, 950.0, 100, 0x4, Not Active, Not Active, Not Active, Active",
        "1980, 2070, 120.0, 10, 0x0, Not Active, Not Active, Active, Not Active",  # idle
        "2070, 2070, 910.0, 99, 0x0, Not Active, Not Active, Not Active, Not Active",
        "[N/A]",
    ]
    s.f.write("\n".join(rows) + "\n")
    rec = s.stop()
    # the idle sample is left out: its reason does not count
    assert rec == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                   "samples": 3}


def _capture_fields():
    text = open(os.path.join(bench.ROOT, "profiles", "score_tc_cfg2_ncu.md")).read()
    return dict((k, v.strip()) for k, v in (line.split(":", 1) for line in text.splitlines()
                if line.startswith(("dram_bytes_per_launch:", "captured_layers:"))))


def test_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    f = _capture_fields()
    full = bench.score_traffic(32)
    if full is not None:   # the committed sources are the captured ones
        assert full == float(f["dram_bytes_per_launch"]) * 32 / float(f["captured_layers"])
    # a copy of the repository whose kernel differs by one byte: no figure
    fake = tmp_path / "repo"
    csrc = fake / "kv_cache_eviction_snapkv_gb300" / "csrc"
    csrc.mkdir(parents=True)
    shutil.copytree(os.path.join(bench.ROOT, "profiles"), fake / "profiles")
    src = os.path.join(bench.ROOT, "kv_cache_eviction_snapkv_gb300", "csrc")
    for name in ("score_tc.cu", "tc_common.cuh"):
        shutil.copy(os.path.join(src, name), csrc / name)
    monkeypatch.setattr(bench, "ROOT", str(fake))
    assert bench.score_traffic(32) == full
    with open(csrc / "score_tc.cu", "a") as fh:
        fh.write("\n")
    assert bench.score_traffic(32) is None


def test_describe_scaling_modes():
    wl = wk.make_workload("cfg2")
    weak, strong = bench.describe(wl), bench.describe(wl, split=True)
    assert "weak" in weak["parallelism"] and "strong" in strong["parallelism"]
    assert weak["instances"] == 32 * 32 and weak["seq_lens"] == [16384]
    assert weak["workload"].startswith("cfg2")
