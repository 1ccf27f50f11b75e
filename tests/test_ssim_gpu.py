"""Parity of the CUDA L1 + SSIM loss and gradient (through the C ABI) with
the oracle: the three image workloads in full, lambda 0 / 0.2 / 1, ragged
and tiny images, identical images, and the loss gradient feeding the
rasterizer's backward.

Tolerances: loss, mean SSIM and mean L1 within 1e-6 absolute (sums done in
double; each SSIM value carries float32 rounding, mostly from the
variance terms E[x^2] - mu^2, whose error ~u E[x^2] is divided by at least
C2 = 9e-4, and these errors average out over the image); gradient elements
within 1e-3 max|dL/dx| (the rasterizer's gradient bar; the same variance
rounding enters the adjoint maps)."""
import numpy as np
import pytest

from synth.images import make_image_pair

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def run():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gaussian_splatting_differentiable_gb300 as ss

    def _run(x, y, lam=0.2):
        C, H, W = x.shape
        sl = ss.SsimLoss(C, H, W, lam, "cuda")
        g = sl(torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda())
        torch.cuda.synchronize()
        return sl.loss.cpu().numpy().astype(np.float64), g.cpu().numpy()
    return _run


def _check(run, x, y, lam=0.2):
    import oracle.ssim as OS
    loss, g = run(x, y, lam)
    o = OS.loss_and_grad(x, y, lam)
    assert abs(loss[0] - o["loss"]) <= 1e-6, (loss, o["loss"])
    assert abs(loss[1] - o["ssim"]) <= 1e-6, (loss, o["ssim"])
    assert abs(loss[2] - o["l1"]) <= 1e-6, (loss, o["l1"])
    t = 1e-3 * np.abs(o["grad"]).max() if np.abs(o["grad"]).max() > 0 else 1e-30
    err = np.abs(g - o["grad"])
    assert err.max() <= t, (err.max(), t, np.unravel_index(err.argmax(), err.shape))
    return {"loss": float(loss[0]), "loss_err": float(abs(loss[0] - o["loss"])),
            "grad_err_over_tol": float(err.max() / t)}


@pytest.mark.parametrize("wl", [21, 22, 23])
def test_workloads(run, wl):
    x, y = make_image_pair(wl)
    print(wl, _check(run, x, y))


@pytest.mark.parametrize("lam", [0.0, 1.0])
def test_lambda_extremes(run, lam):
    x, y = make_image_pair(21, seed=3)
    _check(run, x, y, lam)


@pytest.mark.parametrize("C,H,W", [(1, 1, 1), (1, 5, 3), (2, 33, 65), (3, 31, 97), (4, 70, 40),
                                   (1, 32768, 3), (2, 5, 32768)])
def test_ragged_and_tiny(run, C, H, W):
    x, y = make_image_pair(21, seed=C * 100 + H, C=C, H=H, W=W)
    _check(run, x, y)


def test_identical_images(run):
    x, _ = make_image_pair(21, seed=9)
    loss, g = run(x, x)
    assert abs(loss[0]) < 1e-6 and abs(loss[1] - 1.0) < 1e-6 and loss[2] == 0.0
    assert np.abs(g).max() < 1e-9


def test_loss_gradient_feeds_rasterizer(run):
    """render -> loss gradient -> rasterizer backward, all on the device."""
    import torch
    import synth
    import gaussian_splatting_differentiable_gb300 as ss
    sc = synth.make_scene(2)
    r = ss.Rasterizer(sc.W, sc.H, sc.n, 8 * sc.n, ss.SS_ACCUM_WEIGHT, device="cuda")
    sp = ss.Splats.from_numpy(sc, "cuda")
    r.bin_and_sort(sp)
    r.forward(sp)
    _, tgt = make_image_pair(21, seed=1, C=3, H=sc.H, W=sc.W)
    sl = ss.SsimLoss(3, sc.H, sc.W, 0.2, "cuda")
    g = sl(r.image, torch.from_numpy(tgt).cuda())
    r.backward(sp, g)
    torch.cuda.synchronize()
    assert torch.isfinite(r.grads["dmean2d"]).all()
    assert float(r.grads["drgb"].abs().sum()) > 0
