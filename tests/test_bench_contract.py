"""bench.py's output contract, checked on the host: the reference arm (the
fp64 oracle on the host cores) prints one JSON line with every key the
benchmark contract asks for, and the host-side helpers compute what the
line reports."""
import json
import math
import os
import subprocess
import sys

import bench
from exact_second_order_two_gb300.synthetic import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

REQUIRED = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
            "cpu_baseline", "e2e")


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run(
        [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
         "--workload", "fp32_n256_d64", "--ref-step-seconds", "0.2"],
        cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    for key in REQUIRED:
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["config"]["workload"] == "fp32_n256_d64"
    assert d["value"] > 0 and math.isfinite(d["value"])
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_flop_formula():
    w = WORKLOADS["bf16_causal_b2h16_n16384_d128"]
    # 30 * B*H*N^2*d, halved for the causal mask: 16.49 TFLOP
    assert abs(bench.flops_bob(w) - 30 * 2 * 16 * 16384 ** 2 * 128 / 2) < 1.0
    nc = WORKLOADS["fp32_n256_d64"]
    assert bench.flops_bob(nc) == 30 * 256 ** 2 * 64
    # F_min: the 12 products of a schedule without recomputation
    assert bench.flops_bob(w, 12) == 24 * 2 * 16 * 16384 ** 2 * 128 / 2


def test_warmup_below_three_is_refused():
    out = subprocess.run([sys.executable, "bench.py", "--warmup", "2"], cwd=ROOT,
                         capture_output=True, text=True, timeout=120)
    assert out.returncode != 0


def test_recorded_counters_follow_the_kernel_sources(tmp_path, monkeypatch):
    """The ncu figures in the JSON line (DRAM traffic, shared-memory busy
    fraction) are reported only while the kernel sources still hash to the
    value recorded with the capture."""
    rec = {"wl": {"k": {"bytes_per_launch": 123.0, "smem_tc_pct": 57.0, "smem_lsu_pct": 20.0,
                        "source_hash": "abc"}}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc")
    assert bench.recorded_traffic("k", "wl") == 123.0
    smem = bench.recorded_smem("k", "wl")
    assert abs(smem["total"] - 0.77) < 1e-12 and abs(smem["tensor_core"] - 0.57) < 1e-12
    assert bench.recorded_smem("other", "wl") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "changed")
    assert bench.recorded_traffic("k", "wl") is None and bench.recorded_smem("k", "wl") is None
