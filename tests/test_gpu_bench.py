"""bench.py's own arm on the GPU: one short run at batch 2 prints exactly one JSON
line with the keys its contract names (throughput, latency, roofline of the GEMM
kernel, end-to-end figure with host copies, launch count, clocks)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_bench_line_carries_its_contract_keys():
    steps = 3
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--batch", "2", "--steps", str(steps),
                        "--warmup", "3", "--no-cpu-baseline"], capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["unit"] == "images/s" and d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] == steps
    assert d["ms_per_step"] == pytest.approx(2 * 1e3 / d["value"], rel=1e-6)
    lat = d["latency_ms"]
    assert lat["min"] <= lat["median"] <= lat["max"] and lat["min"] <= lat["mean"] <= lat["max"]
    roof = d["roofline"]
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s" and roof["peak"] > 0
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] == 2 * 378 * 378 * 3 * 2
    assert e2e["d2h_bytes_per_step"] == 2 * 1152 * 2
    # every step launches the same kernels
    assert d["gpu_launches"] > 0 and d["gpu_launches"] % steps == 0
    # a timed region this short may end before the first clock sample
    assert d["clocks"] is None or d["clocks"]["sm_max_mhz"] > 0
