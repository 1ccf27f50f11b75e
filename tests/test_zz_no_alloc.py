"""ss_raster_bwd_noalloc: the backward pass for callers that cannot allocate.

A plugin inside an application that owns all device memory, or a real-time
thread that must not risk the synchronisation cudaMalloc / cudaFree can
cause, cannot give the library a workspace.  ss_raster_bwd_noalloc keeps its
accumulated-weight scratch in a fixed array inside the library instead.  This
checks, through the C ABI, that two calls in a row return what ss_raster_bwd
returns, within the tolerances of the parity tests: the second call also
shows that the array's leftover contents from the first call do not leak.
The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

FIELDS = ("dmean2d", "dconic", "dopacity", "drgb")


@pytest.fixture(scope="module")
def ss():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gaussian_splatting_differentiable_gb300 as m
    return m


def test_noalloc_backward_matches_workspace_backward_twice(ss):
    import torch
    sc = synth.make_scene(2)          # 5,207 splats, 256x256, accumulated weight on
    flags = ss.SS_ACCUM_WEIGHT
    sp = ss.Splats.from_numpy(sc)
    dL = torch.from_numpy(sc.dL_dimage).cuda()
    r = ss.Rasterizer(sc.W, sc.H, sc.n, 4 * sc.n, flags, bg=sc.bg)
    r.bin_and_sort(sp)
    r.forward(sp)
    r.backward(sp, dL)                # ss_raster_bwd, with a workspace
    torch.cuda.synchronize()
    ref = {k: r.grads[k].cpu().numpy().astype(np.float64) for k in FIELDS}
    ref_w = r.accum_weight.cpu().numpy().astype(np.float64)
    assert np.abs(ref_w).max() > 0

    for call in range(2):
        grads = {k: torch.full_like(r.grads[k], float("nan")) for k in FIELDS}
        w = torch.full_like(r.accum_weight, float("nan"))
        ss.ss_raster_bwd_noalloc(r.records, sc.n, r.vals, r.tile_offsets, r.n_pairs, sc.W, sc.H,
                                 sc.bg, flags, r.T_final, r.last_contrib, r.blend_masks, dL,
                                 grads, w)
        torch.cuda.synchronize()
        for k in FIELDS:
            got = grads[k].cpu().numpy().astype(np.float64)
            tol = max(1e-4, 1e-3 * np.abs(ref[k]).max())
            assert np.all(np.abs(got - ref[k]) <= tol), (call, k, np.abs(got - ref[k]).max(), tol)
        got_w = w.cpu().numpy().astype(np.float64)
        tol_w = np.maximum(1e-5, 2.0 ** -23 * np.abs(ref_w))
        assert np.all(np.abs(got_w - ref_w) <= tol_w), (call, np.abs(got_w - ref_w).max())


def test_noalloc_rejects_more_splats_than_its_scratch(ss):
    from gaussian_splatting_differentiable_gb300._lib import SsGrads
    L = ss._L
    big = (1 << 21) + 1
    g = SsGrads(0x1000, 0x1000, 0x1000, 0x1000)
    st = L.ss_raster_bwd_noalloc(0x1000, big, 0x1000, 0x1000, 16, 64, 64, None, 1, 0x1000,
                                 0x1000, 0x1000, 0x1000, ctypes.byref(g), 0x1000, None)
    assert st == 5                     # SS_ERR_UNSUPPORTED, nothing launched
    assert "fixed scratch" in ss.ss_last_error()
