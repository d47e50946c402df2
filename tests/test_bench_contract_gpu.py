"""bench.py's JSON line on a GPU: one short run of the 1024^3 workload (with
the 256^3 workload as its extra-workloads leg) must print every field the
bench contract asks for, with consistent values."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_has_every_contract_field(cuda_device):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "sq1024", "--steps", "5",
           "--warmup", "3", "--e2e-steps", "2", "--extra-workloads", "sq256"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    d = json.loads(lines[0])

    for key, typ in (("metric", str), ("value", float), ("unit", str), ("n_gpus", int), ("steps", int),
                     ("warmup", int), ("ms_per_step", float), ("higher_is_better", bool), ("scaling", str),
                     ("dtype", str), ("data", str), ("config", dict), ("e2e", dict), ("gpu_launches", int),
                     ("roofline", dict), ("cpu_baseline", dict), ("clocks", dict)):
        assert key in d, key
        assert isinstance(d[key], typ) or (typ is float and isinstance(d[key], int)), (key, d[key])
    assert "vs_baseline" in d and d["vs_baseline"] is None
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["value"] > 0
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["dtype"] == "f32"
    assert d["config"]["workload"] == "sq1024"
    assert d["gpu_launches"] >= d["steps"]

    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 2 * 4 * 1024 * 1024 and e2e["d2h_bytes_per_step"] == 4 * 1024 * 1024

    roof = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in roof, key
    assert roof["bound"] == "alu" and roof["unit"] == "TFLOP/s"
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    assert 0 < roof["frac"] < 1.2
    assert roof["achieved_basis"].startswith("2MNK / mean CUDA-event time of one call")
    assert d["gpu_launches"] % d["steps"] == 0   # every step launches the same kernels

    cpu = d["cpu_baseline"]
    for key in ("value", "unit", "cores", "kind", "sample"):
        assert key in cpu, key
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] > 0
    assert isinstance(cpu["cpu_model"], str) and cpu["cpu_model"]

    extra = d["workloads"]
    assert list(extra) == ["sq256"]
    x = extra["sq256"]
    assert x["value"] > 0 and x["unit"] == "GFLOP/s" and x["steps"] >= 5
    assert x["shape"]["M"] == x["shape"]["N"] == x["shape"]["K"] == 256
    assert x["step_ms"]["best"] <= x["step_ms"]["median"]
    assert 0 < x["fp32_peak_pct"] < 120 and x["l2"] == "flushed between steps"
    assert "reasons" in x["clocks"]

    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
