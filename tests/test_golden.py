"""Hand-derived worked examples (tests/golden/closed_forms.json) against the
oracle on the CPU and against the CUDA path on the GPU.

Each case is a one- or two-splat scene whose image, transmittance, last
contributor and nine gradient fields follow in closed form from the model of
2D Gaussian splats composited front to back ("Phase 5 step 30b --
kernel-by-kernel timing": rasterize_f32, rasterize_backwards; the 2D backward
of "从 8.6 KB 到 4.2 KB ..."): the fixture states each derivation next to its
values, written as expressions in exp() so that they can be checked by eye.
No program produced them, so they pin the oracle (and the kernels) to the
mathematics rather than to themselves.
"""
import json
import math
import os

import numpy as np
import pytest

import synth

FIXTURE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "closed_forms.json")
FIELDS = ("dmean2d", "dconic", "dopacity", "drgb")


def _value(expr: str) -> float:
    """A fixture value: a number or an arithmetic expression in exp()."""
    return float(eval(expr, {"__builtins__": {}}, {"exp": math.exp}))


def _cases():
    with open(FIXTURE) as f:
        return json.load(f)["cases"]


def _scene(case) -> synth.Scene:
    W, H, s = case["W"], case["H"], case["splats"]
    f32 = lambda x: np.ascontiguousarray(np.asarray(x, np.float64).astype(np.float32))  # noqa: E731
    dL = np.zeros((3, H, W))
    for x, y, r, g, b in case["dL"]:
        dL[:, y, x] = (r, g, b)
    return synth.Scene(W=W, H=H, mean2d=f32(s["mean2d"]), conic=f32(s["conic"]),
                       opacity=f32(s["opacity"]), rgb=f32(s["rgb"]), depth=f32(s["depth"]),
                       dL_dimage=f32(dL), bg=f32(case["bg"]), accum_weight=True,
                       median_depth=False, name=case["name"])


def _expected_grads(case):
    out = {}
    for k in FIELDS:
        rows = [g[k] for g in case["grads"]]
        out[k] = np.array([[_value(e) for e in (r if isinstance(r, list) else [r])] for r in rows])
    return out


def _check(case, image, T, last, grads, tol_px, grad_tol):
    for p in case["pixels"]:
        x, y = p["x"], p["y"]
        want = [_value(e) for e in p["image"]]
        np.testing.assert_allclose(image[:, y, x], want, rtol=0, atol=tol_px,
                                   err_msg="%s: image at (%d, %d)" % (case["name"], x, y))
        assert abs(float(T[y, x]) - _value(p["T"])) <= tol_px, (case["name"], "T", x, y)
        assert int(last[y, x]) == p["last"], (case["name"], "last", x, y)
    want = _expected_grads(case)
    for k in FIELDS:
        got = np.asarray(grads[k], np.float64).reshape(want[k].shape)
        tol = grad_tol(want[k])
        np.testing.assert_allclose(got, want[k], rtol=0, atol=tol,
                                   err_msg="%s: %s" % (case["name"], k))


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_oracle_matches_worked_example(case):
    import oracle
    sc = _scene(case)
    tl = oracle.tile_lists(sc)
    f = oracle.forward(sc, tl["vals"], tl["offs"])
    g = oracle.backward(sc, tl["vals"], tl["offs"])["grads"]
    # The inputs are float32 (0.9 and 0.995 are not exact there); the
    # oracle works in double from them, so 1e-6 covers the input rounding
    # and nothing more.
    _check(case, f["image"], f["T_final"], f["last"], g, 1e-6, lambda w: 1e-6)


def test_fixture_pins_catch_a_planted_mistake():
    """A wrong expected value fails the comparison (the check is not vacuous):
    the two-splat case with the back splat's opacity gradient halved."""
    case = [c for c in _cases() if c["name"].startswith("two splats")][0]
    case = json.loads(json.dumps(case))
    case["grads"][1]["dopacity"] = "-0.5"
    import oracle
    sc = _scene(case)
    tl = oracle.tile_lists(sc)
    f = oracle.forward(sc, tl["vals"], tl["offs"])
    g = oracle.backward(sc, tl["vals"], tl["offs"])["grads"]
    with pytest.raises(AssertionError):
        _check(case, f["image"], f["T_final"], f["last"], g, 1e-6, lambda w: 1e-6)


@pytest.mark.gpu
@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_cuda_path_matches_worked_example(case):
    import parity
    out = parity.run_gpu(_scene(case))
    # The parity tolerances: 1e-5 on image and T; per gradient field
    # max(1e-4, 1e-3 max|field|).
    _check(case, out["image"], out["T_final"], out["last"], out, 1e-5,
           lambda w: max(1e-4, 1e-3 * float(np.abs(w).max())))
