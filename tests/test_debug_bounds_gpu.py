"""The SS_DEBUG_BOUNDS build: device-side bounds checks that record an error
word and skip or clamp the access they guard, never trap.

The library is built a second time with -DSS_DEBUG_BOUNDS (libss_debug.so)
and loaded in child processes (SS_LIBRARY): workloads 1-3 through the
training step's path, the CUDA graph and the entry points that take the
splats themselves run clean and still match the oracle; a last_contrib made
to reach past its tile's list (which the library clamps, so no access
leaves its buffer) is reported by the debug build and not by the normal one.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def debug_lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "ss_build", os.path.join(ROOT, "gaussian_splatting_differentiable_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build(debug_bounds=True)


def _run(code: str, lib: str | None) -> str:
    env = dict(os.environ)
    if lib:
        env["SS_LIBRARY"] = lib
    else:
        env.pop("SS_LIBRARY", None)
    prog = "import sys\nsys.path.insert(0, %r)\nsys.path.insert(0, %r)\n" % (
        ROOT, os.path.join(ROOT, "tests")) + textwrap.dedent(code)
    r = subprocess.run([sys.executable, "-c", prog], env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    return r.stdout


def test_debug_build_runs_the_workloads_clean(debug_lib):
    out = _run("""
        import synth, parity
        import gaussian_splatting_differentiable_gb300 as ss
        assert ss.ss_debug_bounds_enabled()
        for wl in (1, 2, 3):
            sc = synth.make_scene(wl)
            r = parity.full_parity(sc)
            assert ss.ss_debug_status() == ss.SS_OK, (wl, ss.ss_last_error())
            r = parity.full_parity(sc, graph=True)
            assert ss.ss_debug_status() == ss.SS_OK, (wl, ss.ss_last_error())
            sc.weight_stats = sc.distortion = False
            r = parity.full_parity(sc, path="splats")
            assert ss.ss_debug_status() == ss.SS_OK, (wl, ss.ss_last_error())
            print("workload", wl, "clean")
        print("ok")
    """, debug_lib)
    assert out.strip().endswith("ok")


STALE_LAST = """
    import torch, synth
    import gaussian_splatting_differentiable_gb300 as ss
    sc = synth.make_scene(2)
    sp = ss.Splats.from_numpy(sc)
    dL = torch.from_numpy(sc.dL_dimage).cuda()
    r = ss.Rasterizer(sc.W, sc.H, sc.n, 4 * sc.n, ss.SS_ACCUM_WEIGHT, bg=sc.bg)
    r.bin_and_sort(sp)
    r.forward(sp)
    assert ss.ss_debug_status() == ss.SS_OK
    offs = r.tile_offsets.cpu().numpy()
    r.last_contrib[5, 7] = int(offs[1] - offs[0]) + 5   # pixel (7, 5) is in tile 0
    r.backward(sp, dL)
    st = ss.ss_debug_status()
    print("status", st, ss.ss_last_error())
"""


def test_debug_build_reports_a_last_contrib_past_its_list(debug_lib):
    out = _run(STALE_LAST, debug_lib)
    assert "status %d" % 6 in out and "0x10" in out, out


def test_normal_build_clamps_the_same_input_silently(debug_lib):
    out = _run(textwrap.dedent(STALE_LAST) + "\nassert not ss.ss_debug_bounds_enabled()\n", None)
    assert "status 0" in out, out
