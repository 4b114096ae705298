"""The benchmark's JSON line on CPU: the reference arm (the oracle on the host
cores) prints one line with the keys the contract asks for, and its numbers are
consistent with one another. The GPU arm needs a device and is exercised by the
GPU runs."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_consistent_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                          "--steps", "1", "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600,
                         check=True).stdout.strip().splitlines()
    assert len(out) == 1
    line = json.loads(out[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["unit"] == "TB/s" and line["higher_is_better"] is True
    assert line["config"]["workload"].startswith("tiny_gqa")
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] > 0
    assert line["e2e"] == {"value": line["value"], "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # value is the algorithmic bytes of the call over the per-call time
    import bench
    import workloads as wl

    w = wl.tiny_gqa_f32()
    assert abs(bench.algorithmic_bytes(w) / (line["ms_per_step"] * 1e-3) / 1e12 - line["value"]) <= 1e-9 * line["value"]


def test_step_statistics_and_traffic_lookup():
    import bench

    st = bench.step_stats([0.0601, 0.0603, 0.0602, 0.0900])
    assert st["us_p99_max"][1] == 90.0
    assert abs(st["us_p10_p50_p90"][1] - 60.25) < 1e-9
    # a traffic line counts only while the kernel sources hash to the recorded value
    assert bench.recorded_traffic("decode_mma_kernel", "no_such_workload") is None
    sha = bench.kernel_sha()
    assert len(sha) == 12 and all(c in "0123456789abcdef" for c in sha)
