"""The benchmark's one JSON line: every key the measurement contract names,
with consistent values, for the product arm (on the GPU, tiny workload) and
for the reference arm (the oracle on the host cores, tiny workload)."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _line(args, timeout):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, capture_output=True,
                       text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def _common(d, steps, warmup):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "e2e", "cpu_baseline"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == warmup
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["scaling"] == "weak" and d["data"] == "synthetic"
    assert d["config"]["workload"] == "tiny"
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"]
    assert "h2d_bytes_per_step" in e and "d2h_bytes_per_step" in e
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0 and c["sample"]


def test_reference_arm_line_on_the_host():
    d = _line(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"], 600)
    _common(d, 2, 3)
    assert d["impl"] == "reference" and d["dtype"] == "f64"
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0


@pytest.mark.gpu
def test_product_arm_line_on_the_gpu():
    d = _line(["--workload", "tiny", "--steps", "4", "--warmup", "3", "--repeats", "2", "--no-workloads"], 900)
    _common(d, 4, 3)
    assert d["dtype"] == "bf16" and "impl" not in d
    r = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in r, key
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert d["gpu_launches"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    assert d["parity"]["ok"] and d["parity"]["units"] == d["parity"]["of_units"]
    clk = d["clocks"]
    assert "sm_mhz" in clk and "sm_max_mhz" in clk and "reasons" in clk
