"""Host arithmetic of bench.py's report, on the CPU: the blended-pair count
read from the forward's blend masks and the per-kernel roofline rows."""
import os
import sys

import pytest

torch = pytest.importorskip("torch")
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_blended_pairs_counts_set_bits_of_the_used_columns_only():
    cap, n = 7, 5
    m = torch.zeros(8 * cap, dtype=torch.int32)
    rows = m.view(8, cap)
    rows[0, 0] = 0b1011                       # 3 bits
    rows[3, 4] = -1                           # all 32 bits (0xffffffff)
    rows[7, 2] = -(1 << 31)                   # 1 bit (0x80000000)
    rows[5, 5] = -1                           # past n: not counted
    rows[6, 6] = 0x0f0f                       # past n: not counted
    assert bench.blended_pairs(m, cap, n) == 3 + 32 + 1


def test_kernel_rooflines_divide_the_model_by_the_measured_time():
    steps = 10
    kernels = {
        "k_emit_pairs": {"launches": 10, "ms_total": 0.5},
        "k_sort_hist": {"launches": 10, "ms_total": 0.2},
        "k_sort_pass": {"launches": 60, "ms_total": 3.0},
        "k_sort_final": {"launches": 10, "ms_total": 0.15},
        "k_sort_ties": {"launches": 10, "ms_total": 0.05},
        "k_raster_fwd": {"launches": 10, "ms_total": 4.0},
        "k_raster_bwd": {"launches": 10, "ms_total": 6.0},
    }
    n, P, HW = 1000, 4000, 2000
    hbm, red = 1000.0, 1e10
    rows = bench.kernel_rooflines(kernels, steps, n, P, HW, cand=10 ** 8, active=5 * 10 ** 7,
                                  blended=10 ** 7, hbm=hbm, hbm_src="test", red_rate=red,
                                  accum=True, sms=100, sm_mhz=1000.0)
    b = rows["k_emit_pairs"]
    assert b["algorithmic_bytes"] == 28 * n + 12 * P
    assert b["frac"] == pytest.approx((28 * n + 12 * P) / 0.05e-3 / 1e9 / hbm)
    s = rows["sort (hist, passes, final, ties)"]
    assert s["algorithmic_bytes"] == (24 * 6 + 16) * P        # 6 passes a step
    assert s["ms_per_call"] == pytest.approx(0.34)
    f = rows["k_raster_fwd"]
    lanes = 100 * 128 * 1000e6
    assert f["alu"]["frac"] == pytest.approx(10 ** 8 * 16 / lanes / 0.4e-3)
    assert f["hbm"]["algorithmic_bytes"] == 40 * P + 20 * HW
    k = rows["k_raster_bwd"]
    assert k["hbm"]["algorithmic_bytes"] == 40 * P + 20 * HW + 44 * n
    assert k["l2_atomic"]["atomics"] == 10 * P
    assert k["l2_atomic"]["frac"] == pytest.approx(10 * P / red / 0.6e-3)
    assert k["alu_active"]["frac"] == pytest.approx(5e7 * 47 / lanes / 0.6e-3)
    assert k["alu_blended"]["frac"] == pytest.approx(1e7 * 47 / lanes / 0.6e-3)


def test_issue_and_shared_memory_ceilings_use_the_recorded_counters_only():
    rec = {"inst_executed_per_launch": 4.0e8, "smem_wavefronts_per_launch": 1.0e8}
    sms, mhz, ms = 100, 1000.0, 0.5
    i = bench.issue_ceiling(10 ** 7, ms, sms, mhz, rec["inst_executed_per_launch"])
    assert i["model_ms"] == pytest.approx(1e7 * 31 / 32 / (sms * 4 * mhz * 1e6) * 1e3)
    assert i["issue_frac_if_every_cycle_issued"] == pytest.approx(4e8 / (sms * 4 * 1e9) / 0.5e-3)
    m = bench.smem_ceiling(ms, sms, mhz, rec)
    assert m["model_ms"] == pytest.approx(1e8 / (sms * 1e9) * 1e3)
    assert m["frac"] == pytest.approx((1e8 / (sms * 1e9)) / (ms * 1e-3))
    # a record of another source (None) gives no figure
    assert bench.smem_ceiling(ms, sms, mhz, None)["wavefronts_per_launch"] is None
    assert "frac" not in bench.smem_ceiling(ms, sms, mhz, None)


def test_sort_passes_follow_the_recorded_depth_range():
    import numpy as np
    c = np.zeros(4, np.uint64)
    c[2], c[3] = np.float32(1.0).view(np.uint32), np.float32(100.0).view(np.uint32)
    assert bench.sort_passes(c, 4056) == 5           # 12 tile bits + 26 depth bits
    c[3] = np.float32(1e30).view(np.uint32)
    assert bench.sort_passes(c, 4056) == 6           # all 32 depth bits
    c[2], c[3] = np.float32(3.0).view(np.uint32), np.float32(3.0).view(np.uint32)
    assert bench.sort_passes(c, 16) == 3             # 16-bit floor + 4 tile bits
    c[2], c[3] = np.uint64(2 ** 64 - 1), 0           # no pairs: the full key
    assert bench.sort_passes(c, 4056) == 6


def _last_json_line(out: str) -> dict:
    import json
    lines = [l for l in out.splitlines() if l.startswith("{")]
    assert lines, out[-2000:]
    return json.loads(lines[-1])


def test_reference_arm_prints_the_contract_line():
    """bench.py --impl reference times the oracle on the host cores and prints
    one JSON line with the arm's fields (tiny workload, a second or so)."""
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "1",
                        "--steps", "3", "--warmup", "3"], cwd=root, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = _last_json_line(r.stdout)
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0
    # the timed steps are one whole step, measured, not extrapolated
    assert abs(d["whole_step_ms"] - d["ms_per_step"] * d["steps"]) <= 1e-6 * d["whole_step_ms"]
    assert abs(d["value"] * d["whole_step_ms"] * 1e-3 - d["config"]["candidate_splat_px"]) <= \
        1e-6 * d["config"]["candidate_splat_px"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
