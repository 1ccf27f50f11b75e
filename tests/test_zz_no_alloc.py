"""ss_raster_bwd_noalloc: the backward pass for callers that cannot allocate.

A plugin inside an application that owns all device memory, or a real-time
thread that must not risk the synchronisation cudaMalloc / cudaFree can
cause, cannot give the library a workspace.  ss_raster_bwd_noalloc keeps its
accumulated-weight scratch in a fixed array inside the library instead.
These tests call it through the C ABI and check, within the tolerances of
the parity tests:
  * two calls in a row against ss_raster_bwd_records and against the oracle, with
    and without the accumulated weight (the second call also shows that the
    array's leftover contents from the first do not leak);
  * a third call on a smaller scene after the larger ones (each call clears
    only its own prefix of the array);
  * the 2M-splat scene, inside the array's 2,097,152-splat limit, against
    the oracle;
  * that a first call on a stream being captured is refused cleanly (in a
    fresh process, where nothing has looked the array up yet).
The file is named to be collected last.
"""
import ctypes
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

FIELDS = ("dmean2d", "dconic", "dopacity", "drgb")
P_DIST = "ddepth"


@pytest.fixture(scope="module")
def ss():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gaussian_splatting_differentiable_gb300 as m
    return m


def _prepared(ss, sc, flags):
    """Splats binned, sorted and composited by the workspace path; the
    workspace backward's gradients as the reference."""
    import torch
    sp = ss.Splats.from_numpy(sc)
    dL = torch.from_numpy(sc.dL_dimage).cuda()
    r = ss.Rasterizer(sc.W, sc.H, sc.n, 4 * sc.n, flags, bg=sc.bg)
    r.bin_and_sort(sp)
    r.forward(sp)
    r.backward(sp, dL)                # ss_raster_bwd_records, with a workspace
    torch.cuda.synchronize()
    ref = {k: r.grads[k].cpu().numpy().astype(np.float64) for k in FIELDS}
    ref_w = r.accum_weight.cpu().numpy().astype(np.float64) if r.accum_weight is not None else None
    return r, dL, ref, ref_w


def _noalloc(ss, r, sc, flags, dL):
    """One ss_raster_bwd_noalloc call into NaN-filled outputs; numpy copies."""
    import torch
    grads = {k: torch.full_like(r.grads[k], float("nan")) for k in FIELDS}
    w = torch.full((sc.n,), float("nan"), dtype=torch.float32, device="cuda")
    ss.ss_raster_bwd_noalloc(r.records, sc.n, r.vals, r.tile_offsets, r.n_pairs, sc.W, sc.H,
                             sc.bg, flags, r.T_final, r.last_contrib, r.blend_masks, dL, grads,
                             w if flags & ss.SS_ACCUM_WEIGHT else None)
    torch.cuda.synchronize()
    out = {k: v.cpu().numpy() for k, v in grads.items()}
    out["accum"] = w.cpu().numpy() if flags & ss.SS_ACCUM_WEIGHT else None
    out[P_DIST] = None
    return out


def _against_workspace_path(out, ref, ref_w, what):
    for k in FIELDS:
        got = out[k].astype(np.float64)
        tol = max(1e-4, 1e-3 * np.abs(ref[k]).max())
        assert np.all(np.abs(got - ref[k]) <= tol), (what, k, np.abs(got - ref[k]).max(), tol)
    if ref_w is not None:
        got_w = out["accum"].astype(np.float64)
        tol_w = np.maximum(1e-5, 2.0 ** -23 * np.abs(ref_w))
        assert np.all(np.abs(got_w - ref_w) <= tol_w), (what, np.abs(got_w - ref_w).max())


def _against_oracle(sc, out):
    import oracle
    import parity
    tl = oracle.tile_lists(sc)
    obw = oracle.backward(sc, tl["vals"], tl["offs"], threads=oracle.default_threads())
    return parity.check_backward(sc, out, obw)


@pytest.mark.parametrize("accum", [True, False], ids=["accum", "no-accum"])
def test_noalloc_backward_twice_then_a_smaller_scene(ss, accum):
    flags = ss.SS_ACCUM_WEIGHT if accum else 0
    sc = synth.make_scene(2)           # 5,207 splats, 256 x 256
    sc.accum_weight = accum
    r, dL, ref, ref_w = _prepared(ss, sc, flags)
    if accum:
        assert np.abs(ref_w).max() > 0
    for call in range(2):
        out = _noalloc(ss, r, sc, flags, dL)
        _against_workspace_path(out, ref, ref_w, "call %d" % call)
        print("call", call, _against_oracle(sc, out))
    small = synth.make_scene(1)        # 256 splats: a prefix of what the calls above used
    small.accum_weight = accum
    r2, dL2, ref2, ref2_w = _prepared(ss, small, flags)
    out = _noalloc(ss, r2, small, flags, dL2)
    _against_workspace_path(out, ref2, ref2_w, "smaller scene")
    print("smaller scene", _against_oracle(small, out))


def test_noalloc_full_size_scene_against_the_oracle(ss):
    """The 2M-splat scene (inside the array's 2,097,152-splat limit), with the
    accumulated weight, against the oracle over every splat."""
    sc = synth.make_scene(4)
    flags = ss.SS_ACCUM_WEIGHT
    r, dL, ref, ref_w = _prepared(ss, sc, flags)
    out = _noalloc(ss, r, sc, flags, dL)
    _against_workspace_path(out, ref, ref_w, "2M splats")
    print("2M splats", _against_oracle(sc, out))


def test_noalloc_rejects_more_splats_than_its_scratch(ss):
    from gaussian_splatting_differentiable_gb300._lib import SsGrads
    L = ss._L
    big = (1 << 21) + 1
    g = SsGrads(0x1000, 0x1000, 0x1000, 0x1000)
    st = L.ss_raster_bwd_noalloc(0x1000, big, 0x1000, 0x1000, 16, 64, 64, None, 1, 0x1000,
                                 0x1000, 0x1000, 0x1000, ctypes.byref(g), 0x1000, None)
    assert st == 5                     # SS_ERR_UNSUPPORTED, nothing launched
    assert "fixed scratch" in ss.ss_last_error()


def test_noalloc_first_call_while_capturing_is_refused(ss):
    """In a fresh process, where nothing has looked the array up: a first call
    made on a stream being captured returns SS_ERR_UNSUPPORTED (the capture
    is left intact and ends normally); the next call outside the capture
    works."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = textwrap.dedent("""
        import sys, torch
        sys.path.insert(0, %r)
        import synth
        import gaussian_splatting_differentiable_gb300 as ss
        sc = synth.make_scene(1)
        sp = ss.Splats.from_numpy(sc)
        dL = torch.from_numpy(sc.dL_dimage).cuda()
        r = ss.Rasterizer(sc.W, sc.H, sc.n, 4 * sc.n, ss.SS_ACCUM_WEIGHT, bg=sc.bg)
        r.bin_and_sort(sp)
        r.forward(sp)
        torch.cuda.synchronize()
        args = (r.records, sc.n, r.vals, r.tile_offsets, r.n_pairs, sc.W, sc.H, sc.bg,
                ss.SS_ACCUM_WEIGHT, r.T_final, r.last_contrib, r.blend_masks, dL, r.grads,
                r.accum_weight)
        g = torch.cuda.CUDAGraph()
        status = None
        with torch.cuda.graph(g):
            try:
                ss.ss_raster_bwd_noalloc(*args)
            except ss.SSError as e:
                status = e.status
        print("capture status", status, ss.ss_last_error())
        assert status == 5, status
        ss.ss_raster_bwd_noalloc(*args)
        torch.cuda.synchronize()
        assert float(r.accum_weight.abs().max()) > 0
        print("ok")
    """ % root)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    print(res.stdout, res.stderr[-2000:])
    assert res.returncode == 0 and "ok" in res.stdout
