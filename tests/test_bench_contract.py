"""bench.py's output line, checked on the CPU through the reference arm (the CPU oracle,
which needs no GPU): one JSON line with every key of the benchmark contract, for the
same metric and workload as the GPU arm, and consistent numbers."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stdout + p.stderr
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    return json.loads(lines[0])


def test_reference_arm_line_has_every_contract_key():
    line = _run("--impl", "reference", "--steps", "3", "--warmup", "3")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["steps"] == 3 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["scaling"] == "weak" and line["vs_baseline"] is None
    assert line["value"] > 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    # the same workload, metric and config object as the GPU arm
    import bench
    assert line["metric"] == bench.METRIC
    assert line["config"] == bench.config_block("full", 1, bench.FULL_STEP_BYTES)
    assert line["config"]["bytes_per_step"] == bench.FULL_STEP_BYTES
    # a step is one sample step, actually timed: value and ms_per_step describe it, and
    # the timed steps fit in the measured wall time of the timed region
    assert line["sample_bytes_per_step"] * bench.SAMPLE_DIV == bench.FULL_STEP_BYTES
    assert abs(line["value"] - line["sample_bytes_per_step"] / (line["ms_per_step"] / 1e3) / 1e9) \
        <= 1e-3 * line["value"] + 1e-4
    assert line["steps"] * line["ms_per_step"] / 1e3 <= line["wall_s_timed_region"] * 1.01
    assert cb["cores"] == cb["host"]["cpu_count"]


import pytest  # noqa: E402


@pytest.mark.gpu
def test_gpu_arm_line_has_every_contract_key():
    """The GPU arm on the small workload (the same code path as the full one): roofline,
    clocks, launch count and the end-to-end figure with its copied bytes."""
    line = _run("--workload", "small", "--steps", "3", "--warmup", "3", "--no-cpu-baseline")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "clocks", "gpu_launches", "e2e"):
        assert key in line, key
    assert line["value"] > 0 and line["n_gpus"] == 1 and line["steps"] == 3
    rf = line["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) <= 1e-3
    assert 0.3 < rf["frac"] < 1.2
    assert rf["traffic"] is None        # the stored DRAM traffic is the full workload's
    ck = line["clocks"]
    assert ck["sm_mhz"] > 0 and ck["sm_max_mhz"] > 0 and isinstance(ck["reasons"], list)
    assert line["gpu_launches"] == 5 * line["steps"]     # AdamW, 2 softmax, LayerNorm rows + columns
    ks = line["kernels"]
    assert set(ks) == {"adamw", "softmax_f32", "softmax_bf16", "layernorm_bf16"}
    assert ks["adamw"]["timing"] == "in step"
    bw = line["backward_in_step"]
    assert bw["ms"] > 0 and bw["bytes"] == sum(ks[n]["bytes"] for n in ks if n != "adamw")
    # the backward kernels timed alone add up to about their share of the step
    assert 0.7 < bw["sum_of_back_to_back_ms"] / bw["ms"] < 1.3
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    link = e2e["link"]
    assert link["h2d_ms"] > 0 and link["d2h_ms"] > 0 and link["both_ms"] > 0
    # (the rate was computed before the milliseconds were rounded to 0.01)
    assert abs(link["h2d_GB_s"] - e2e["h2d_bytes_per_step"] / link["h2d_ms"] / 1e6) \
        <= 0.005 * link["h2d_GB_s"] + 0.1
    # the floor is the slower of the two-way copies and the device step; no loop beats it
    assert e2e["floor_ms"] >= link["both_ms"] - 0.01 and e2e["floor_ms"] >= line["ms_per_step"] - 0.01
    assert 0 < e2e["frac_of_floor"] <= 1.05
    assert abs(e2e["frac_of_floor"] - e2e["floor_ms"] / e2e["step_ms"]) <= 2e-3


@pytest.mark.gpu
def test_hidden_size_sweep_lines():
    """bench.py --sweep-hidden: one JSON line per op and shape with a consistent
    bandwidth figure; with --sweep-reps 0 it only calls each shape once."""
    args = [sys.executable, os.path.join(ROOT, "bench.py"), "--sweep-hidden", "--sweep-shapes",
            "bf16:1004,bf16:4096,f32:6144", "--sweep-mb", "16"]
    p = subprocess.run(args + ["--sweep-reps", "2"], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert p.returncode == 0, p.stdout + p.stderr
    lines = [json.loads(ln) for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert [(d["op"], d["dtype"], d["D"]) for d in lines] == [
        (op, dt, D) for dt, D in (("bf16", 1004), ("bf16", 4096), ("f32", 6144))
        for op in ("layernorm_bwd", "rmsnorm_bwd")]
    for d in lines:
        es = 4 if d["dtype"] == "f32" else 2
        assert d["rows"] == (16 << 20) // (d["D"] * es)
        assert d["us"] > 0 and 0 < d["frac"] < 1.5
        peak = float(d["peak"].split()[0])
        assert abs(d["frac"] * peak - d["GB_s"]) <= 0.0006 * peak + 0.1   # frac has 3 decimals
    p = subprocess.run(args + ["--sweep-reps", "0"], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert p.returncode == 0, p.stdout + p.stderr
    assert not [ln for ln in p.stdout.splitlines() if ln.startswith("{")]


@pytest.mark.gpu
def test_causal_sweep_lines():
    """bench.py --sweep-causal: one JSON line per dtype and S, rows in whole S x S blocks,
    consistent bandwidth figures; with --sweep-reps 0 it only calls each shape once."""
    args = [sys.executable, os.path.join(ROOT, "bench.py"), "--sweep-causal", "--sweep-shapes",
            "bf16:1024,f32:512,bf16:4096", "--sweep-mb", "8"]
    p = subprocess.run(args + ["--sweep-reps", "2"], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert p.returncode == 0, p.stdout + p.stderr
    lines = [json.loads(ln) for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert [(d["dtype"], d["S"]) for d in lines] == [("bf16", 1024), ("f32", 512), ("bf16", 4096)]
    for d in lines:
        es = 4 if d["dtype"] == "f32" else 2
        S = d["S"]
        assert d["rows"] == S * max(1, (8 << 20) // (S * S * es))
        assert d["us"] > 0 and 0 < d["frac"] < 1.5 and 0 < d["dense_frac"] < 1.5
        peak = float(d["peak"].split()[0])
        assert abs(d["frac"] * peak - d["GB_s"]) <= 0.0006 * peak + 0.1
    p = subprocess.run(args + ["--sweep-reps", "0"], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert p.returncode == 0, p.stdout + p.stderr
    assert not [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
