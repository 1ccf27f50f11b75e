"""Parity of the CUDA projection (forward and backward, through the C ABI)
against the projection oracle: the three projection workloads (the 2M-splat
one at full size, compared on 20,000 sampled splats: each splat's outputs
depend on that splat alone), every SH degree, ragged counts, culled splats of
every kind, and the projection feeding the rasterizer and back."""
import numpy as np
import pytest

from synth.scene3d import make_scene3d

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def PP():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import parity_project
    return parity_project


@pytest.mark.parametrize("wl", [11, 12])
def test_workload_full_parity(PP, wl):
    r = PP.full_parity(make_scene3d(wl))
    print("workload", wl, r)
    assert r["culled"] > 0


def test_two_million_splats_sampled(PP):
    r = PP.sampled_parity(make_scene3d(13))
    print(r)


@pytest.mark.parametrize("deg", [0, 1, 2, 3])
def test_sh_degrees(PP, deg):
    PP.full_parity(make_scene3d(11, seed=2, n=3000, sh_degree=deg))


@pytest.mark.parametrize("n", [1, 255, 257, 1000])
def test_ragged_counts(PP, n):
    PP.full_parity(make_scene3d(11, seed=3, n=n))


def test_culled_kinds(PP):
    sc = make_scene3d(11, seed=4, n=300)
    c = -(np.asarray(sc.cam.R, np.float64).T @ np.asarray(sc.cam.t, np.float64))
    sc.mean3[0] = c.astype(np.float32)                   # at the camera centre
    sc.mean3[1, 2] = np.float32(-2.0)                    # behind
    sc.quat[2] = 0.0                                     # rotation undefined
    sc.scale[3] = 0.0                                    # degenerate: blur keeps it valid
    sc.mean3[4] = np.float32([np.inf, 0, 5])             # non-finite
    sc.sh[:, 0, 5] = np.float32(-10.0)                   # red clamped to 0
    r = PP.full_parity(sc)
    assert r["culled"] >= 4


def test_zero_splats(PP):
    import torch
    import gaussian_splatting_differentiable_gb300 as ss
    sc = make_scene3d(11, n=0)
    sp = ss.Splats3D.from_numpy(sc, "cuda")
    pr = ss.Projector(0, 3, "cuda")
    pr.forward(sp, PP.cam_struct(sc.cam))
    e = torch.empty(0, device="cuda")
    pr.backward(sp, PP.cam_struct(sc.cam), e, e, e)
    torch.cuda.synchronize()


def test_projection_feeds_rasterizer_and_back(PP):
    """project -> bin / sort / fwd / bwd -> project backward on the device;
    the 3D gradients equal the oracle's projection backward applied to the
    rasterizer's 2D gradients."""
    import torch
    import gaussian_splatting_differentiable_gb300 as ss
    import oracle.project as OP
    sc = make_scene3d(11, seed=6, n=2000, W=128, H=96)
    dev = torch.device("cuda")
    sp3 = ss.Splats3D.from_numpy(sc, dev)
    cam = PP.cam_struct(sc.cam)
    pr = ss.Projector(sc.n, sc.sh_degree, dev)
    pr.forward(sp3, cam)
    opacity = torch.from_numpy(sc.opacity).to(dev)
    r = ss.Rasterizer(sc.W, sc.H, sc.n, 64 * sc.n, ss.SS_ACCUM_WEIGHT, device=dev)
    dL = torch.from_numpy(np.random.default_rng(0).normal(0, 0.1, (3, sc.H, sc.W))
                          .astype(np.float32)).to(dev)
    splats = pr.splats2d(opacity)
    r.step(splats, dL)
    assert int((r.last_contrib > 0).sum()) > 1000
    pr.backward(sp3, cam, r.grads["dmean2d"], r.grads["dconic"], r.grads["drgb"])
    torch.cuda.synchronize()
    up = {k: r.grads[k].cpu().numpy() for k in ("dmean2d", "dconic", "drgb")}
    gpu = {k: v.cpu().numpy() for k, v in pr.grads.items()}
    ob = OP.project_backward(sc, upstream=up)
    for k in PP.FIELDS3:
        ref, got = ob[k], gpu[k]
        t = max(1e-4, 1e-3 * np.abs(ref).max())
        assert np.abs(got - ref).max() <= t, k
