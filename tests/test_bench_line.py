"""The benchmark's JSON line: the keys and the relations between them that the
measurement contract fixes, on the tiny workload (reference arm on the CPU;
the GPU arm on a GPU)."""
import json
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent


def _run(*args, timeout=600):
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), *args], capture_output=True, text=True,
                       timeout=timeout, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _run("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1")
    assert d["impl"] == "reference" and d["higher_is_better"] is True and d["dtype"] == "f64"
    assert d["steps"] == 2 and d["warmup"] == 1 and d["config"]["workload"] == "tiny"
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


@pytest.mark.gpu
def test_gpu_arm_line(gpu):
    d = _run("--workload", "tiny", "--extra", "llama8b", "--steps", "5", "--warmup", "3", "--warm-ms", "50")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks", "cpu_baseline",
              "stats", "max_abs_err"):
        assert k in d, k
    assert d["steps"] == 5 and d["n_gpus"] == 1 and d["scaling"] == "weak" and d["config"]["workload"] == "tiny"
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert d["gpu_launches"] == 5  # one fused launch per step
    assert d["max_abs_err"] is not None and d["max_abs_err"] <= 5e-3
    assert d["stats"]["n"] >= 50 and d["stats"]["p10_ms"] <= d["stats"]["median_ms"] <= d["stats"]["p90_ms"]
    e = d["e2e"]
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] == 4 * 4 * 128 * 4
    w = d["per_workload"]["llama8b"]
    assert w["config"]["workload"] == "llama8b" and w["max_abs_err"] <= 5e-3 and w["roofline"]["frac"] > 0.5
