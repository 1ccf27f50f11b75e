"""bench.py's own arm on a tiny workload: the JSON line carries every field
of the contract (the driver reads these), with the roofline, the per-kernel
rooflines, the end-to-end figure and the launch count."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_bench_line_has_the_contract_fields():
    r = subprocess.run([sys.executable, "bench.py", "--workload", "1", "--steps", "3",
                        "--warmup", "3", "--no-next", "--no-cpu-baseline"], cwd=ROOT,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    d = json.loads(lines[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
              "e2e", "gpu_launches", "clocks", "kernel_rooflines"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert d["config"]["workload"] == "tiny-64x64-256"
    ro = d["roofline"]
    assert ro["bound"] == "hbm" and ro["unit"] == "GB/s" and ro["peak"] > 0
    assert ro["frac"] == pytest.approx(ro["achieved"] / ro["peak"])
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] >= 10 * 3
    assert set(d["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    kr = d["kernel_rooflines"]
    assert {"k_emit_pairs", "k_raster_fwd", "k_raster_bwd"} <= set(kr)
