"""The benchmark's JSON line keeps its contract: one line on stdout with the
keys the measurement harness reads, for the library's arm (on a GPU) and for
the reference arm (the oracle, on the host cores, no GPU needed)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
COMMON = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
          "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e",
          "cpu_baseline")


def run_bench(*args, timeout=900):
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=timeout)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, res.stdout
    return json.loads(lines[0])


def test_reference_arm_line():
    d = run_bench("--impl", "reference", "--steps", "1", "--warmup", "1")
    for k in COMMON + ("impl",):
        assert k in d, k
    assert d["impl"] == "reference" and "unavailable" not in d
    assert d["value"] > 0 and d["unit"] == "frame pairs/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "3840x2160_16bit_x32"


@pytest.mark.gpu
def test_library_arm_line():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = run_bench("--steps", "5", "--warmup", "3", "--no-cpu", "--no-e2e")
    for k in COMMON + ("roofline", "clocks", "gpu_launches"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] >= 3
    assert d["scaling"] == "weak" and d["data"] == "synthetic"
    assert d["config"]["workload"] == "3840x2160_16bit_x32" and "l2" in d["config"]
    r = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and 0 < r["frac"] < 1.5
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    for k in ("sm_mhz", "sm_max_mhz", "reasons"):
        assert k in d["clocks"], k
    # two launches a step (the fused pass and the per-frame sums)
    assert d["gpu_launches"] == 2 * d["steps"]
    # the median of repeated regions, with its spread
    t = d["timing"]
    assert t["repeats"] >= 21
    assert t["region_ms"]["min_ms"] <= t["region_ms"]["median_ms"] <= t["region_ms"]["max_ms"]
    assert abs(d["ms_per_step"] - t["region_ms"]["median_ms"] / d["steps"]) < 1e-9
    # the other measured configurations, timed in the same run
    from exact_full_reference_gb300 import workloads as wl

    assert sorted(d["configs"]) == sorted(c for c in wl.BENCH_CONFIGS if c != wl.HEADLINE)
    for name, c in d["configs"].items():
        assert c["value"] > 0 and c["repeats"] >= 21 and 0 < c["kernel_frac"] < 1.5, name
