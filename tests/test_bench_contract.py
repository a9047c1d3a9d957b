"""bench.py's reference arm (the float64 oracle on the host) prints one JSON
line with the keys the benchmark contract names, and --gpus N agrees with the
number of ranks a launcher started; no GPU involved."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                         text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _run("--impl", "reference", "--workload", "single_256x128", "--steps", "2", "--warmup", "1")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == "steps/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 1
    assert abs(d["ms_per_step"] - 1000.0 / d["value"]) <= 1e-6 * d["ms_per_step"]
    assert d["config"]["workload"] == "single_256x128"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_gpus_flag_and_world_size_agree():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.launch_plan(1, {}) == "run"
    assert bench.launch_plan(8, {}) == "relaunch"                       # N ranks started by bench.py itself
    assert bench.launch_plan(4, {"WORLD_SIZE": "4"}) == "run"           # started by torchrun with N ranks
    assert bench.launch_plan(1, {"WORLD_SIZE": "1"}) == "run"
    for gpus, env in ((8, {"WORLD_SIZE": "1"}), (1, {"WORLD_SIZE": "2"}), (0, {})):
        plan = bench.launch_plan(gpus, env)
        assert plan not in ("run", "relaunch") and plan


def test_mismatched_world_size_exits_nonzero():
    env = dict(os.environ, WORLD_SIZE="3", RANK="0", LOCAL_RANK="0")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--workload",
                          "single_256x128", "--no-cpu-baseline"], cwd=ROOT, capture_output=True, text=True,
                         timeout=600, env=env)
    assert out.returncode != 0
    assert "WORLD_SIZE=3" in out.stderr


def test_l2_note_follows_the_workload():
    # the timed steps do not flush L2: a line says whether its inputs exceed it
    sys.path.insert(0, ROOT)
    import bench
    import muonh_workloads as wl
    assert bench._l2_note(wl.qwen3_2b(), "muonh").startswith("inputs larger than L2")
    assert bench._l2_note(wl.batched_256(), "muonh").startswith("inputs larger than L2")
    assert bench._l2_note(wl.single_256x128(), "muonh").startswith("inputs fit in L2")


def test_traffic_figure_names_its_workload():
    # the roofline's DRAM traffic is reported only for the workload it was captured on
    with open(os.path.join(ROOT, "profiles", "ns_gemm_traffic.json")) as f:
        d = json.load(f)
    assert d["workload"] == "qwen3_2b_28layers"
    assert 1e9 < d["bytes_per_launch"] < 1e10
    assert os.path.exists(os.path.join(ROOT, "profiles", d["source"].split(":")[0]))
