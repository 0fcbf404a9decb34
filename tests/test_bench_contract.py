"""bench.py's one-line JSON contract, run end to end on the tiny workload.

The reference arm (the oracle on the host cores) runs on the CPU; the main
line, the MXFP8 format and the side-stream sweep need the GPU.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
             "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def test_reference_arm_line():
    d = run_bench("--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "0")
    assert BASE_KEYS <= set(d), set(d)
    assert d["config"]["experts_per_step"] >= 1 and "experts" in d["cpu_baseline"]["sample"]
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"].startswith("tiny")


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", ["deepseek", "mxfp8", "per_tensor"])
def test_main_line(fmt):
    d = run_bench("--config", "tiny", "--steps", "5", "--warmup", "3", "--no-cpu-baseline",
                  "--format", fmt, "--records", "v2lite")
    assert (BASE_KEYS - {"cpu_baseline"}) <= set(d), set(d)
    assert d["value"] > 0 and d["steps"] == 5 and d["warmup"] == 3 and d["n_gpus"] == 1
    r = d["roofline"]
    assert {"bound", "achieved", "peak", "unit", "frac", "traffic"} <= set(r)
    assert r["bound"] in ("tensor", "hbm") and 0 < r["frac"] < 2
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0 and d["gpu_launches"] % d["steps"] == 0
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    assert {"median", "p10", "p90"} <= set(d["step_ms"])
    assert d["l2_warm"]["ms_per_step"] > 0 and d["l2_warm"]["steps"] >= 1
    assert "idle" in d["config"]["timing"]          # the settled power state is stated
    assert d["config"]["format"].startswith("MXFP8" if fmt == "mxfp8" else "E4M3")
    assert ("per-tensor" in d["config"]["format"]) == (fmt == "per_tensor")
    lr = d["layer_roofline"]
    assert lr["fp8_peak"] == "2 x measured bf16 burst" and 0 < lr["fp8_peak_frac"] < 2
    # the per-workload record: the same timing method on another workload
    rec = d["per_workload"]["records"]["v2lite"]
    assert rec["workload"].startswith("dsv2lite") and rec["steps"] == 5 and rec["ms_per_step"] > 0
    assert {"fc1", "fc2", "combine"} <= set(rec["kernel_ms"]) and 0 < rec["layer_roofline"]["frac"] < 2


@pytest.mark.gpu
def test_side_stream_sweep_line():
    d = run_bench("--config", "tiny", "--side-mlp", "256", "--steps", "3", "--warmup", "1",
                  "--no-cpu-baseline")
    assert d["unit"] == "ms" and d["higher_is_better"] is False
    assert d["layer_ms"] > 0 and d["mlp_ms"] > 0 and d["serial_ms"] > 0
    assert len(d["concurrent"]) >= 2 and all(p["ms"] > 0 for p in d["concurrent"])


@pytest.mark.parametrize("name,touched,gb", [
    ("v2lite", 64, 0.5875),      # every expert routed
    ("v3prefill", 256, 11.512),
    ("v3decode8", 52, 2.29),     # the experts seed 0 touches at T = 8
])
def test_layer_roofline_bytes(name, touched, gb):
    """The layer roofline's compulsory bytes: FP8 weights and scales of every
    routed expert, x and out in BF16, the routes; experts with no route cost
    nothing."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    from gen import configs
    wl = configs.WORKLOADS[name]
    counts = np.zeros(wl.E, np.int64)
    counts[:touched] = 1
    b, t = bench.algorithmic_bytes(wl, counts)
    assert t == touched
    per_expert = 3 * wl.I * wl.H + (2 * wl.I // 128 + wl.I // 128) * (wl.H // 128) * 4
    assert b == touched * per_expert + wl.T * wl.H * 4 + wl.T * wl.K * 8
    assert abs(b / 1e9 - gb) < 0.01 * gb


def test_oracle_sample_is_every_row_of_its_experts():
    """A bounded oracle sample is every routed row of the experts it draws:
    the mini-problem keeps exactly those routes (others masked) and its FLOPs
    count 6*H*I per kept row."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    from gen import configs, problem
    wl = configs.TINY
    idx, w = wl.make_routes()
    smp = bench.OracleSampler(wl, problem.x_bits(wl), idx, w)
    dt, fl, rows, n = smp.sample(3, np.random.default_rng(5))
    assert n == 3 and dt > 0
    counts = np.bincount(idx.ravel(), minlength=wl.E)
    assert rows in {int(counts[list(s)].sum()) for s in __import__("itertools").combinations(range(wl.E), 3)}
    assert fl == 6 * rows * wl.H * wl.I
