"""bench.py's GPU arm prints the one JSON line its readers parse (GPU): every
key, with the roofline object of the dominant kernel, the end-to-end leg, the
oracle's CPU baseline, the clock record of the timed region and the secondary
e4m3-scores line."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_small_workload_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "small",
                          "--steps", "5", "--warmup", "3", "--cpu-seconds", "2"],
                         cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-3000:]
    d = json.loads([l for l in out.stdout.splitlines() if l.strip()][-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e",
              "gpu_launches", "roofline", "cpu_baseline", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] >= 3
    assert d["value"] > 0 and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["config"]["workload"].startswith("small")
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert 0 < r["frac"] < 1.5 and r["achieved"] > 0 and r["peak"] > 0
    assert "traffic" in r
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["value"] > 0 and c["cores"] >= 1 and c["sample"]
    k = d["clocks"]
    assert k["sm_max_mhz"] and "reasons" in k
    assert len(d["peak_hbm_gb_by_tiles_per_chunk"]) == 2  # memory at two tile sizes
    e8 = d["e4m3_scores"]  # the secondary line with the score products on e4m3
    assert e8["dtype"] == "bf16+e4m3" and e8["value"] > 0 and e8["unit"] == d["unit"]
