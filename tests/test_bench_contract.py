"""Both arms of the benchmark print the one JSON line the measurement contract
asks for: the reference arm (the oracle timed on the host cores, on a tiny
sample: one (b, kv-head) pair, one step) with the same metric and workload as
the GPU arm, and the GPU arm on a short run."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1", "--cpu-pairs", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    sys.path.insert(0, ROOT)
    import bench
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "steps/s" and line["higher_is_better"] is True
    assert line["config"]["workload"] == bench.WORKLOAD["workload"]
    assert line["steps"] == 1 and line["warmup"] == 1 and line["n_gpus"] == 1
    assert line["value"] > 0 and abs(line["ms_per_step"] - 1000.0 / line["value"]) < 1e-6 * line["ms_per_step"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["h2d_bytes_per_step"] == 0


@pytest.mark.gpu
def test_gpu_arm_prints_the_contract_line():
    """The GPU arm on a short run (4 layers, 3 timed steps) prints one JSON line
    with every key of the measurement contract, its roofline of the dominant
    call, the end-to-end figure, the clocks and the launch count."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--layers", "4", "--steps", "3",
                        "--warmup", "3", "--no-cpu-baseline", "--no-configs"], capture_output=True, text=True,
                       timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "clocks", "gpu_launches"):
        assert key in line, key
    assert line["steps"] == 3 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["value"] > 0 and abs(line["ms_per_step"] - 1000.0 / line["value"]) < 1e-6 * line["ms_per_step"]
    roof = line["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in roof, key
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and 0 < roof["frac"] == roof["achieved"] / roof["peak"]
    # the roofline follows from its own numbers, and the dominant call fits in the timed step
    assert abs(roof["achieved"] * roof["avg_launch_ms"] * 1e6 - roof["algorithmic_bytes_per_launch"]) \
        <= 1e-6 * roof["algorithmic_bytes_per_launch"]
    assert 4 * roof["avg_launch_ms"] <= line["ms_per_step"] * 1.02
    ov = line["overlap"]
    assert ov["steps_per_s_with_prefetch"] > 0 and ov["steps_per_s_staging_preloaded"] > 0
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(line["clocks"])
    assert line["gpu_launches"] > 0 and line["gpu_launches"] % (3 * 4) == 0  # whole launches per layer and step
    # the pre-fetch keeps the rows already staged: a fraction of the rows, and the host bytes below the total
    pr = line["prefetch_rows"]
    assert 0.0 <= pr["kept"] <= 1.0 and 0.0 <= pr["kept_fresh_queries"] <= 1.0
    assert ov["prefetch_host_bytes_per_step"] <= ov["prefetch_bytes_per_step"]


@pytest.mark.gpu
def test_config_point_measures_every_call():
    """One configuration point (configuration 1) through the bench's per-call
    timing: every call of the layer's decode step has a time, bytes and an HBM
    fraction, and the oracle's time on the same layer is beside them."""
    sys.path.insert(0, ROOT)
    import bench
    pts = bench.measure_config(bench.CONFIGS["c1"], 6000.0, oracle_on=True, reps=3)
    assert len(pts) == 1
    pt = pts[0]
    for key in ("decode_step_graph_us", "merged_us", "attn2_us", "topk_us", "gather_us", "quantize_us",
                "merged_bytes", "merged_hbm_frac", "oracle_ms_per_layer"):
        assert pt[key] > 0, key
