"""Pins of the oracle's float32 error model against an emulated float32
evaluation of the rasterizer's arithmetic.

The oracle composites in double and flags a decision as a knife edge when a
float32 evaluation could take it the other way (the alpha floor, the alpha
cap, the termination, the median's T = 0.5); the parity tolerances of the
accumulated weight and of the depth distortion come from the same model.
Here the rasterizer's arithmetic is evaluated in float32 with numpy, in its
order of operations: every + - * rounded to float32, fused multiply-adds
rounded once (the exact product in double, one rounding), and the
hardware approximations -- the base-2 exponential (relative error at most
2^-22), log2f (at most 1 ulp) and the reciprocal (at most 1 ulp) -- taken
as their correctly rounded values pushed to the ends of their documented
error bounds.  On inputs placed at the thresholds, each test checks

  * soundness: every float32 error lies inside the oracle's bound, and
    every decision that flips is one the oracle flags;
  * tightness: the bound is within a stated factor of the largest error
    observed, so it is not vacuous.

The planted mistakes at the end scale each bound up or down and show that a
pin fails.
"""
import math
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import synth

F = np.float32
D = np.float64
LOG2E = F(1.4426950408889634)
KA = F(-0.5) * LOG2E          # the record's -log2(e) / 2 (exact halving of a float32)
KB = -LOG2E
U = 2.0 ** -24
EX2_DOC = 2.0 ** -22          # documented relative error of the hardware 2^x
LN2 = math.log(2.0)


def fma32(a, b, c):
    """a b + c rounded once (the product of two float32 is exact in double)."""
    return (np.asarray(a, D) * np.asarray(b, D) + np.asarray(c, D)).astype(F)


def e2_f32(a, b, c, mx, my, px, py):
    """The rasterizer's base-2 exponent: record coefficients A, B, C as
    float32 products, rounded differences, two products, two fused
    multiply-adds."""
    A, B, C = KA * a, KB * b, KA * c
    dx, dy = F(px) - mx, F(py) - my
    t = fma32(A, dx, B * dy)
    return fma32(dx, t, (C * dy) * dy)


def thr_variants(o):
    """-log2f(fl(255 o)): the correctly rounded value and its two neighbours
    (log2f is within 1 ulp)."""
    p = F(255.0) * o
    thr = -(np.log2(p.astype(D)).astype(F))
    return [np.nextafter(thr, F(-np.inf)), thr, np.nextafter(thr, F(np.inf))]


def ex2_f32(e2, eps):
    """2^e2 with relative error eps (|eps| <= 2^-22), rounded to float32."""
    return (np.exp2(np.asarray(e2, D)) * (1.0 + eps)).astype(F)


def exact_sigma(a, b, c, dx, dy):
    a, b, c, dx, dy = (np.asarray(v, D) for v in (a, b, c, dx, dy))
    return 0.5 * (a * dx * dx + c * dy * dy) + b * dx * dy


def random_splats(rng, n, s_lo, s_hi, o_lo, o_hi):
    th = rng.uniform(0.0, math.pi, n)
    s1 = np.exp(rng.uniform(math.log(s_lo), math.log(s_hi), n))
    s2 = np.exp(rng.uniform(math.log(s_lo), math.log(s_hi), n))
    conic = synth.conic_from_scales(th, s1, s2).astype(F)
    o = rng.uniform(o_lo, o_hi, n).astype(F)
    return conic[:, 0], conic[:, 1], conic[:, 2], o


def at_radius(rng, a, b, c, sig):
    """Float32 means and pixel centres whose offset lies where the exponent
    is sig (before the float32 rounding of the mean), in a random direction."""
    n = a.size
    phi = rng.uniform(0.0, 2 * math.pi, n)
    cs, sn = np.cos(phi), np.sin(phi)
    q = a.astype(D) * cs * cs + 2 * b.astype(D) * cs * sn + c.astype(D) * sn * sn
    r = np.sqrt(2.0 * sig / q)
    px = rng.integers(0, 32, n) + 0.5
    py = rng.integers(0, 32, n) + 0.5
    return (px - r * cs).astype(F), (py - r * sn).astype(F), px, py


# ---------------------------------------------------------------- alpha floor

@pytest.fixture(scope="module")
def floor_samples():
    rng = np.random.default_rng(101)
    n = 400_000
    a, b, c, o = random_splats(rng, n, 0.3, 8.0, 1.02 / 255.0, 1.0)
    sig = np.log(255.0 * o.astype(D)) * (1.0 + rng.uniform(-2e-6, 2e-6, n))
    mx, my, px, py = at_radius(rng, a, b, c, sig)
    dx, dy = px - mx.astype(D), py - my.astype(D)
    s = exact_sigma(a, b, c, dx, dy)
    e2x, thrx = -s / LN2, -np.log2(255.0 * o.astype(D))
    e2f = e2_f32(a, b, c, mx, my, px, py)
    thr = thr_variants(o)
    skip_m, val_m = oracle.margins_n(a, b, c, dx, dy, o)
    oG = o.astype(D) * np.exp(-s)
    return dict(e2f=e2f, thr=thr, e2x=e2x, thrx=thrx, skip_m=skip_m, val_m=val_m, oG=oG)


def test_floor_decision_error_inside_skip_margin(floor_samples):
    """ln 2 (|e2 error| + |thr error|), the largest change of ln(255 alpha)
    a float32 evaluation can make, never exceeds the oracle's skip margin;
    every flipped decision is flagged."""
    S = floor_samples
    need = LN2 * (np.abs(S["e2f"].astype(D) - S["e2x"]) +
                  np.max([np.abs(t.astype(D) - S["thrx"]) for t in S["thr"]], axis=0))
    assert np.all(need * (1.0 + 2.0 * need) <= S["skip_m"]), np.max(need / S["skip_m"])
    keep = S["oG"] >= 1.0 / 255.0
    flipped = np.zeros_like(keep)
    for t in S["thr"]:
        flipped |= (S["e2f"] >= t) != keep
    flagged = np.abs(S["oG"] - 1.0 / 255.0) <= S["skip_m"] * S["oG"]
    assert flipped.sum() > 1000, "the samples do not reach the knife-edge band"
    assert np.all(flagged[flipped])


def test_floor_margin_is_tight(floor_samples):
    """The skip margin is within 2x of the largest error seen, and small in
    absolute terms (the median margin at the threshold is below 5e-6)."""
    S = floor_samples
    need = LN2 * (np.abs(S["e2f"].astype(D) - S["e2x"]) +
                  np.max([np.abs(t.astype(D) - S["thrx"]) for t in S["thr"]], axis=0))
    assert np.max(need / S["skip_m"]) >= 0.5
    assert np.median(S["skip_m"]) < 5e-6
    flagged = np.abs(S["oG"] - 1.0 / 255.0) <= S["skip_m"] * S["oG"]
    keep = S["oG"] >= 1.0 / 255.0
    flipped = np.zeros_like(keep)
    for t in S["thr"]:
        flipped |= (S["e2f"] >= t) != keep
    # the flagged band is at most a few times wider than the band of flips
    assert flagged.sum() <= 12 * flipped.sum()


# ---------------------------------------------------------------- alpha value and cap

def _value_errors(a, b, c, o, mx, my, px, py):
    dx, dy = px - mx.astype(D), py - my.astype(D)
    s = exact_sigma(a, b, c, dx, dy)
    oGx = o.astype(D) * np.exp(-s)
    e2f = e2_f32(a, b, c, mx, my, px, py)
    outs = [(o * ex2_f32(e2f, eps)) for eps in (-EX2_DOC, 0.0, EX2_DOC)]
    err = np.max([np.abs(v.astype(D) / oGx - 1.0) for v in outs], axis=0)
    skip_m, val_m = oracle.margins_n(a, b, c, dx, dy, o)
    return err, val_m, oGx, outs


def test_alpha_value_error_inside_value_margin():
    """The relative error of the float32 o 2^e2 (the exponent's error, the
    exponential's 2^-22, one rounding) never exceeds the value margin, over
    the whole blended range of exponents; the margin is within 3x of the
    largest error seen."""
    rng = np.random.default_rng(102)
    n = 300_000
    a, b, c, o = random_splats(rng, n, 0.3, 8.0, 0.02, 1.0)
    sig = rng.uniform(0.0, 1.0, n) * np.log(255.0 * o.astype(D))
    mx, my, px, py = at_radius(rng, a, b, c, sig)
    err, val_m, _, _ = _value_errors(a, b, c, o, mx, my, px, py)
    assert np.all(err <= val_m), np.max(err / val_m)
    assert np.max(err / val_m) >= 0.35


def test_alpha_cap_flips_are_flagged():
    """Near o G = 0.99 the float32 cap decision (o G > 0.99f) flips only
    where the oracle flags a cap knife edge."""
    rng = np.random.default_rng(103)
    n = 300_000
    a, b, c, _ = random_splats(rng, n, 0.3, 8.0, 0.5, 0.6)
    o = rng.uniform(0.9905, 1.0, n).astype(F)
    sig = np.log(o.astype(D) / 0.99) * (1.0 + rng.uniform(-3e-4, 3e-4, n))
    mx, my, px, py = at_radius(rng, a, b, c, sig)
    err, val_m, oGx, outs = _value_errors(a, b, c, o, mx, my, px, py)
    assert np.all(err <= val_m)
    capped = oGx > 0.99
    flipped = np.zeros_like(capped)
    for v in outs:
        flipped |= (v > F(0.99)) != capped
    flagged = np.abs(oGx - 0.99) <= val_m * 0.99
    assert flipped.sum() > 100
    assert np.all(flagged[flipped])


# ---------------------------------------------------------------- transmittance chains

def _chain_scene(seed, n=2500, W=32, H=32):
    wl = synth.Workload("chains", W, H, n, (0.5, 6.0), (0.02, 0.6), (1.0, 50.0), 0.1, True, True)
    return synth.make_scene(wl, seed=seed)


def emulate_forward(sc, tl, eps_ex2=0.0, thr_pick=1, dist=False, tiles=None):
    """The rasterizer's forward per pixel in float32 (tile by tile, pixels as
    vectors): blend decisions, T, last contributor, median depth, the
    blended steps' alpha and T before, and (dist) the distortion by the
    running totals relative to the first blended depth.  tiles: only these
    tile ids (default all)."""
    W, H = sc.W, sc.H
    tx, ty = oracle.tiles_xy(W, H)
    a, b, c = (np.ascontiguousarray(sc.conic[:, k]) for k in range(3))
    mx, my, o, z = sc.mean2d[:, 0], sc.mean2d[:, 1], sc.opacity, sc.depth
    thr_all = thr_variants(o)[thr_pick]
    out = {"T": np.ones((H, W), F), "last": np.zeros((H, W), np.int64),
           "median": np.zeros((H, W), F), "dist": np.zeros((H, W), F), "steps": {}}
    offs = tl["offs"].astype(np.int64)
    for t in (range(tx * ty) if tiles is None else tiles):
        x0, y0 = 16 * (t % tx), 16 * (t // tx)
        ys, xs = np.mgrid[y0:min(y0 + 16, H), x0:min(x0 + 16, W)]
        xs, ys = xs.ravel(), ys.ravel()
        px, py = (xs + 0.5).astype(F), (ys + 0.5).astype(F)
        m = xs.size
        T = np.ones(m, F)
        done = np.zeros(m, bool)
        last = np.zeros(m, np.int64)
        med = np.zeros(m, F)
        dA, dD1, dD2, dD, zref = (np.zeros(m, F) for _ in range(5))
        steps = [[] for _ in range(m)]
        for k, i in enumerate(tl["vals"][offs[t]:offs[t + 1]]):
            e2 = e2_f32(a[i], b[i], c[i], mx[i], my[i], px, py)
            alpha = np.minimum(F(0.99), o[i] * ex2_f32(e2, eps_ex2))
            Tn = T * (F(1.0) - alpha)
            cand = ~done & (e2 >= thr_all[i])
            stop = cand & (Tn < F(1e-4))
            blend = cand & ~stop
            done |= stop
            if not blend.any():
                continue
            w = alpha * T
            med = np.where(blend & (T > F(0.5)), z[i], med)
            if dist:
                zref = np.where(blend & (dA == F(0.0)), z[i], zref)
                zz = z[i] - zref
                dD = np.where(blend, fma32(w, fma32(zz, fma32(zz, dA, F(-2.0) * dD1), dD2), dD), dD)
                dA = np.where(blend, dA + w, dA)
                dD1 = np.where(blend, fma32(w, zz, dD1), dD1)
                dD2 = np.where(blend, fma32(w * zz, zz, dD2), dD2)
            for p in np.nonzero(blend)[0]:
                steps[p].append((k, float(alpha[p]), float(T[p])))
            T = np.where(blend, Tn, T)
            last = np.where(blend, k + 1, last)
        out["T"][ys, xs] = T
        out["last"][ys, xs] = last
        out["median"][ys, xs] = med
        out["dist"][ys, xs] = dD
        for p in range(m):
            out["steps"][(int(xs[p]), int(ys[p]))] = steps[p]
    return out


@pytest.fixture(scope="module")
def chains():
    sc = _chain_scene(7)
    tl = oracle.tile_lists(sc)
    traces = {(x, y): oracle.trace_pixel(sc, tl["vals"], tl["offs"], x, y)
              for y in range(sc.H) for x in range(sc.W)}
    ofw = oracle.forward(sc, tl["vals"], tl["offs"])
    emus = [emulate_forward(sc, tl, eps, pick) for eps, pick in
            ((0.0, 1), (EX2_DOC, 2), (-EX2_DOC, 0))]
    return sc, tl, traces, ofw, emus


def test_transmittance_error_inside_relT(chains):
    """Along every pixel's chain of ~50-150 blends, the float32 T before each
    blended splat and the final T stay within the oracle's relT bound; a
    pixel whose float32 blend set differs is flagged at the first differing
    position, with the floor, cap or termination kind."""
    sc, tl, traces, ofw, emus = chains
    worst, compared, flipped = 0.0, 0, 0
    for emu in emus:
        for key, tr in traces.items():
            got = emu["steps"][key]
            pos = [s[0] for s in got]
            if pos != list(tr["rec"]["pos"]):
                flipped += 1
                assert any(k in (oracle.AMB_ALPHA, oracle.AMB_CLAMP, oracle.AMB_TERM)
                           for _, k in tr["amb"]), (key, tr["amb"])
                continue
            for (k, al, Tf), r in zip(got, tr["rec"]):
                e = abs(Tf / r["T"] - 1.0)
                assert e <= r["relT"] + 1e-15, (key, k, e, r["relT"])
                if r["relT"] > 0:
                    worst = max(worst, e / r["relT"])
            Tf = float(emu["T"][key[1], key[0]])
            assert abs(Tf / tr["T_final"] - 1.0) <= tr["relT"], key
            compared += 1
    assert compared > 0.99 * len(emus) * len(traces)
    # with the exponential biased to one end of its error bound the errors
    # add up along the chain: the bound is within 5x of the largest one
    assert worst >= 0.2, worst


def test_median_flips_are_flagged(chains):
    """The median's decision (T before blending > 0.5f) differs between float32
    and double only at pixels the oracle flags with the median kind."""
    sc, tl, traces, ofw, emus = chains
    for emu in emus:
        diff = np.argwhere(emu["median"] != ofw["median"].astype(F))
        for (y, x) in diff:
            tr = traces[(int(x), int(y))]
            assert any(k == oracle.AMB_MEDIAN for _, k in tr["amb"]) or \
                list(tr["rec"]["pos"]) != [s[0] for s in emu["steps"][(int(x), int(y))]], (x, y)


# ---------------------------------------------------------------- accumulated weight

def emulate_accum(sc, tl, fwd, rcp_ulps=0):
    """The backward's accumulated weight in float32: per pixel the replay
    T <- T fl(1/fl(1 - alpha)) from the forward's float32 T_final (the
    reciprocal moved by rcp_ulps ulps), w = alpha T; per (8x4 block, splat)
    the float32 sum of its 32 pixels as two interleaved halves; the 32.32
    fixed-point conversion; exact integer sums; the float32 output."""
    W, H = sc.W, sc.H
    tx, _ = oracle.tiles_xy(W, H)
    vals = tl["vals"]
    offs = tl["offs"].astype(np.int64)
    wsum = {}
    for (x, y), steps in fwd["steps"].items():
        T = F(fwd["T"][y, x])
        t = (y // 16) * tx + x // 16
        blk = (t, ((y % 16) // 4) * 2 + (x % 16) // 8)
        lane = (y % 4) * 8 + (x % 8)
        for k, al, _ in reversed(steps):
            al = F(al)
            om = F(1.0) - al
            inv = F(1.0 / float(om))
            for _ in range(abs(rcp_ulps)):
                inv = np.nextafter(inv, F(np.inf) if rcp_ulps > 0 else F(-np.inf))
            Ti = T * inv
            w = al * Ti
            T = Ti
            wsum.setdefault((blk, int(vals[offs[t] + k])), {})[lane] = w
    acc = np.zeros(sc.n, np.uint64)
    for (blk, i), lanes in wsum.items():
        h0, h1 = F(0.0), F(0.0)
        for j in range(16):
            h0 = h0 + lanes.get(2 * j, F(0.0))
            h1 = h1 + lanes.get(2 * j + 1, F(0.0))
        tot = h0 + h1
        acc[i] += np.uint64(np.rint(float(tot * F(4294967296.0))))
    return (acc.astype(D) / 4294967296.0).astype(F)


def test_accumulated_weight_error_inside_accum_err(chains):
    """The float32 evaluation of the accumulated weight differs from the
    oracle's double sum by at most the oracle's accum_err (plus the final
    float32 rounding), with the reciprocal at either end of its 1 ulp; the
    bound is within 7x of the largest error seen."""
    sc, tl, traces, ofw, emus = chains
    obw = oracle.backward(sc, tl["vals"], tl["offs"], slack=True)
    ref, bound = obw["grads"]["accum"], obw["accum_err"]
    worst = 0.0
    for emu in emus:
        same = all([s[0] for s in emu["steps"][key]] == list(tr["rec"]["pos"])
                   for key, tr in traces.items())
        for ulps in (-1, 0, 1):
            got = emulate_accum(sc, tl, emu, ulps).astype(D)
            err = np.abs(got - ref)
            tol = bound + 2.0 ** -24 * np.abs(ref) + (0 if same else obw["slack"]["accum"])
            assert np.all(err <= tol), (np.argmax(err / np.maximum(tol, 1e-300)),
                                        np.max(err / np.maximum(tol, 1e-300)))
            used = ref > 0
            worst = max(worst, float(np.max(err[used] / bound[used])))
    assert worst >= 0.15, worst


# ---------------------------------------------------------------- distortion

def test_distortion_error_inside_dist_err():
    """The float32 distortion by running totals relative to the first blended
    depth differs from the oracle's double sum over pairs by at most the
    oracle's dist_err, on the tiles of workload 3 (depths over [1, 50], up
    to ~100 blends a pixel) where the totals' accumulated rounding is
    largest; the bound is within 10x of the largest error seen there."""
    sc = synth.make_scene(3)
    tl = oracle.tile_lists(sc)
    tx, ty = oracle.tiles_xy(sc.W, sc.H)
    tiles = sorted({(py // 16 + dy) * tx + px // 16 + dx
                    for px, py in ((678, 467), (275, 227), (677, 466), (233, 123))
                    for dy in (-1, 0, 1) for dx in (-1, 0, 1)})
    mask = np.zeros(tx * ty, np.uint8)
    mask[tiles] = 1
    ofw = oracle.forward(sc, tl["vals"], tl["offs"], tile_mask=mask, alt_capacity=1 << 20)
    flagged = np.zeros(sc.W * sc.H, bool)
    flagged[ofw["alts"]["pixel"]] = True
    flagged = flagged.reshape(sc.H, sc.W)
    pix = np.repeat(np.repeat(mask.reshape(ty, tx), 16, 0), 16, 1)[:sc.H, :sc.W].astype(bool)
    worst = 0.0
    for eps, pick in ((0.0, 1), (EX2_DOC, 2), (-EX2_DOC, 0)):
        emu = emulate_forward(sc, tl, eps, pick, dist=True, tiles=tiles)
        same = pix & (emu["last"] == ofw["last"]) & ~flagged
        err = np.abs(emu["dist"].astype(D) - ofw["dist"])
        assert np.all(err[same] <= ofw["dist_err"][same]), np.max(err[same] / ofw["dist_err"][same])
        used = same & (ofw["dist_err"] > 0)
        worst = max(worst, float(np.max(err[used] / ofw["dist_err"][used])))
    assert worst >= 0.1, worst


# ---------------------------------------------------------------- slack

def test_slack_is_the_difference_of_the_two_outcomes():
    """At a pixel where one splat's alpha is 1/255 within 1e-9, the oracle's
    slack (|alternative - normal| contribution per splat and field) equals
    the change of the gradients when the splat's opacity is moved by
    +-1e-7 relative, which takes the decision each way in double."""
    s = 2.0
    o = 0.5
    r = s * math.sqrt(2 * math.log(255 * float(np.float32(o))))
    mean = [[0.5 + r, 10.5], [3.0, 10.0], [1.5, 11.0]]
    conic = [[1 / s**2, 0, 1 / s**2], [0.3, 0.05, 0.2], [0.5, -0.1, 0.4]]
    op = [o, 0.6, 0.4]
    rgb = [[0.9, 0.2, 0.1], [0.1, 0.8, 0.3], [0.2, 0.3, 0.9]]
    depth = [2.0, 1.0, 3.0]
    g = np.random.default_rng(5).normal(0, 1, (3, 32, 32))
    f32 = lambda v: np.ascontiguousarray(np.asarray(v, D).astype(F))  # noqa: E731
    sc = synth.Scene(W=32, H=32, mean2d=f32(mean), conic=f32(conic), opacity=f32(op),
                     rgb=f32(rgb), depth=f32(depth), dL_dimage=f32(g), bg=f32([0, 0, 0]),
                     accum_weight=True, median_depth=False)
    tl = oracle.tile_lists(sc)
    base = oracle.backward(sc, tl["vals"], tl["offs"])
    assert base["slack"]["dopacity"][0] > 0
    # the opacity that puts alpha exactly on 1/255 at pixel (0, 10), moved
    # 1e-9 each way
    a, b, c = sc.conic[0].astype(D)
    dx, dy = 0.5 - float(sc.mean2d[0, 0]), 10.5 - float(sc.mean2d[0, 1])
    alpha0 = float(sc.opacity[0]) * math.exp(-exact_sigma(a, b, c, dx, dy))
    grads = []
    for side in (1.0 + 1e-9, 1.0 - 1e-9):
        fct = side / (255.0 * alpha0)
        p = {"opacity": sc.opacity.astype(D) * np.array([fct, 1.0, 1.0])}
        grads.append(oracle.backward(sc, tl["vals"], tl["offs"], params=p, slack=False)["grads"])
    for k in ("dmean2d", "dconic", "dopacity", "drgb", "accum"):
        diff = np.abs(grads[0][k] - grads[1][k])
        scale = np.abs(base["grads"][k]).max()
        np.testing.assert_allclose(diff, base["slack"][k], rtol=1e-3, atol=1e-5 * scale,
                                   err_msg=k)
        assert base["slack"][k].max() > 0.0, k


# ---------------------------------------------------------------- knife-edge fraction

@pytest.mark.parametrize("wl", [1, 2, 3])
def test_knife_edges_below_a_ten_thousandth_of_the_pixels(wl):
    """Pixels with a knife-edge decision that can change a compared output
    (floor, cap, termination; the median's T = 0.5 only where the median is
    an output) stay below 1e-4 of the pixels on workloads 1-3."""
    sc = synth.make_scene(wl)
    tl = oracle.tile_lists(sc)
    f = oracle.forward(sc, tl["vals"], tl["offs"], alt_capacity=1 << 20,
                       threads=oracle.default_threads())
    kinds = [oracle.AMB_ALPHA, oracle.AMB_TERM, oracle.AMB_CLAMP] + \
        ([oracle.AMB_MEDIAN] if sc.median_depth else [])
    alts = f["alts"]
    px = np.unique(alts["pixel"][np.isin(alts["kind"], kinds)])
    assert px.size < 1e-4 * sc.W * sc.H, (px.size, sc.W * sc.H)


# ---------------------------------------------------------------- planted mistakes

MUTATIONS = [
    ("skip margin x100", "return FIRST_ORDER * U32 * (7.0 * tau + 2.0 * fabs(l) + 1.0);",
     "return 100.0 * FIRST_ORDER * U32 * (7.0 * tau + 2.0 * fabs(l) + 1.0);"),
    ("skip margin / 4", "return FIRST_ORDER * U32 * (7.0 * tau + 2.0 * fabs(l) + 1.0);",
     "return 0.25 * FIRST_ORDER * U32 * (7.0 * tau + 2.0 * fabs(l) + 1.0);"),
    ("value margin x100", "return FIRST_ORDER * (7.0 * U32 * tau + EX2_REL + 1.5 * U32);",
     "return 100.0 * FIRST_ORDER * (7.0 * U32 * tau + EX2_REL + 1.5 * U32);"),
    ("value margin / 4", "return FIRST_ORDER * (7.0 * U32 * tau + EX2_REL + 1.5 * U32);",
     "return 0.25 * FIRST_ORDER * (7.0 * U32 * tau + EX2_REL + 1.5 * U32);"),
    ("relT without the rounding terms", "r->relT += rel_om + U32;",
     "r->relT += alpha * mrel / (1.0 - alpha);"),
    ("accum_err / 8", "accum_err[i] += c1[NF * k + F_W] * relw + 1.0 / 4294967296.0;",
     "accum_err[i] += 0.125 * (c1[NF * k + F_W] * relw + 1.0 / 4294967296.0);"),
    ("accum_err x100", "accum_err[i] += c1[NF * k + F_W] * relw + 1.0 / 4294967296.0;",
     "accum_err[i] += 100.0 * (c1[NF * k + F_W] * relw + 1.0 / 4294967296.0);"),
    ("dist_err / 16", "        *err = e;", "        *err = e / 16.0;"),
    ("slack halved", "d[fld] = byp2[NF * q + fld] - byp1[NF * q + fld];",
     "d[fld] = 0.5 * (byp2[NF * q + fld] - byp1[NF * q + fld]);"),
]


def _run_mutant(tmp_dir, idx, old, new):
    here = os.path.dirname(oracle.__file__)
    src = open(os.path.join(here, "oracle.c")).read()
    if src.count(old) != 1:
        return "pattern"
    d = os.path.join(tmp_dir, "e%02d" % idx)
    os.makedirs(d)
    with open(os.path.join(d, "oracle.c"), "w") as f:
        f.write(src.replace(old, new))
    with open(os.path.join(d, "oracle.h"), "w") as f:
        f.write(open(os.path.join(here, "oracle.h")).read())
    lib = os.path.join(d, "libmut.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", lib,
                    os.path.join(d, "oracle.c"), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not slow", os.path.abspath(__file__)], env=env,
                       capture_output=True, text=True, cwd=os.path.dirname(here))
    return r.returncode


@pytest.fixture(scope="module")
def mutant_results(tmp_path_factory):
    import concurrent.futures as cf
    tmp = str(tmp_path_factory.mktemp("error_model_mutants"))
    workers = max(1, min(len(MUTATIONS), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        futs = [ex.submit(_run_mutant, tmp, i, old, new)
                for i, (_, old, new) in enumerate(MUTATIONS)]
        return [f.result() for f in futs]


@pytest.mark.slow
@pytest.mark.parametrize("k", range(len(MUTATIONS)), ids=[m[0] for m in MUTATIONS])
def test_planted_error_model_mistake_is_caught(mutant_results, k):
    label = MUTATIONS[k][0]
    assert mutant_results[k] != "pattern", "mutation '%s' does not match oracle.c" % label
    assert mutant_results[k] != 0, "planted mistake '%s' passed every pin" % label
