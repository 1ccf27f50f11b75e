"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks the oracle against something it does not compute the same
way: closed forms of one or two splats, compositing invariants, a brute force
over all splats that ignores tiles, an ellipse AABB found by sampling, the
C/Python library sort, and central finite differences of the loss.  The
planted-mistake test at the end shows that plausible slips in oracle.c fail
at least one of these pins.
"""
import math
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import synth

ALPHA_MIN = 1.0 / 255.0


def scene_of(W, H, mean, conic, opacity, rgb, depth, dL=None, bg=(0, 0, 0)):
    n = len(opacity)
    f32 = lambda x: np.ascontiguousarray(np.asarray(x, np.float64).astype(np.float32))  # noqa
    return synth.Scene(W=W, H=H, mean2d=f32(np.reshape(mean, (n, 2))),
                       conic=f32(np.reshape(conic, (n, 3))), opacity=f32(opacity),
                       rgb=f32(np.reshape(rgb, (n, 3))), depth=f32(depth),
                       dL_dimage=f32(np.zeros((3, H, W)) if dL is None else dL),
                       bg=f32(bg), accum_weight=True, median_depth=True)


def render(sc, **kw):
    tl = oracle.tile_lists(sc)
    return tl, oracle.forward(sc, tl["vals"], tl["offs"], **kw)


# ---------------------------------------------------------------- constants / ln

def test_constants():
    c = oracle.constants()
    assert c == {"alpha_min": 1.0 / 255.0, "alpha_max": 0.99, "T_eps": 1e-4, "tile": 16}


def test_ln_series_against_libm():
    xs = np.concatenate([np.geomspace(1.0, 1e6, 4001), [1.0, 2.0, 255.0, 1.5, 3.0, 254.99]])
    for x in xs.astype(np.float32):
        got = oracle.ln(float(x))
        ref = math.log(float(x))
        assert abs(got - ref) <= 1e-6 + 4e-7 * abs(ref), (x, got, ref)


# ---------------------------------------------------------------- binning

def _ellipse_aabb(conic, k):
    """Half widths of {d : d^T Q d <= k} by sampling its boundary (eigh of Q)."""
    a, b, c = conic
    lam, V = np.linalg.eigh(np.array([[a, b], [b, c]], np.float64))
    phi = np.linspace(0, 2 * np.pi, 20001)
    pts = V @ (np.sqrt(k / lam)[:, None] * np.stack([np.cos(phi), np.sin(phi)]))
    return np.abs(pts[0]).max(), np.abs(pts[1]).max()


def test_rect_is_the_alpha_ellipse_aabb():
    """The binning rectangle covers, and is not much larger than, the tiles of
    the AABB of the region where alpha >= 1/255 is possible."""
    sc = synth.make_scene(3, seed=7, n=400, W=600, H=400)
    checked = 0
    for i in range(sc.n):
        st, r = oracle.splat_rect(sc, i)
        o = float(sc.opacity[i])
        k = 2 * math.log(255 * o)
        rx, ry = _ellipse_aabb(sc.conic[i].astype(np.float64), k)
        mx, my = sc.mean2d[i].astype(np.float64)
        tx1, ty1 = oracle.tiles_xy(sc.W, sc.H)
        lo_x = max(0, math.floor((mx - rx) / 16)); hi_x = min(tx1 - 1, math.floor((mx + rx) / 16))
        lo_y = max(0, math.floor((my - ry) / 16)); hi_y = min(ty1 - 1, math.floor((my + ry) / 16))
        if lo_x > hi_x or lo_y > hi_y:
            continue
        assert st == 1
        # covers the exact AABB's tiles
        assert r[0] <= lo_x and r[1] <= lo_y and r[2] >= hi_x and r[3] >= hi_y, (i, r)
        # within the AABB grown by 1 %
        g = 1.01
        assert r[0] >= max(0, math.floor((mx - g * rx - 0.02) / 16))
        assert r[2] <= min(tx1 - 1, math.floor((mx + g * rx + 0.02) / 16))
        assert r[1] >= max(0, math.floor((my - g * ry - 0.02) / 16))
        assert r[3] <= min(ty1 - 1, math.floor((my + g * ry + 0.02) / 16))
        checked += 1
    assert checked > 300


def _alpha_grid(sc, i, x0, y0, w, h):
    ys, xs = np.mgrid[y0:y0 + h, x0:x0 + w]
    dx = xs + 0.5 - float(sc.mean2d[i, 0])
    dy = ys + 0.5 - float(sc.mean2d[i, 1])
    a, b, c = sc.conic[i].astype(np.float64)
    return np.minimum(0.99, float(sc.opacity[i]) * np.exp(-(0.5 * (a * dx * dx + c * dy * dy) + b * dx * dy)))


@pytest.mark.parametrize("wl,n,W,H", [(1, 256, 64, 64), (2, 1500, 256, 256), (3, 600, 200, 120)])
def test_binning_brute_force_over_all_tiles(wl, n, W, H):
    """Every tile holding a pixel centre where a splat reaches alpha >= 1/255
    has that splat's pair; every pair belongs to a valid splat's rectangle."""
    sc = synth.make_scene(wl, seed=3, n=n, W=W, H=H)
    keys, vals, count, culled = oracle.bin_tiles(sc)
    assert count == keys.size and culled == 0
    tx, ty = oracle.tiles_xy(W, H)
    have = set(zip((keys >> np.uint64(32)).tolist(), vals.tolist()))
    assert len(have) == count  # no duplicate pairs
    need = 0
    for i in range(sc.n):
        al = _alpha_grid(sc, i, 0, 0, W, H)
        hit = al >= ALPHA_MIN
        for t in range(tx * ty):
            y0, x0 = (t // tx) * 16, (t % tx) * 16
            if hit[y0:y0 + 16, x0:x0 + 16].any():
                need += 1
                assert (t, i) in have, (i, t)
    assert need <= count <= 4 * need + 10


def test_binning_culls_invalid_splats():
    base = dict(mean=[[8, 8]] * 7, conic=[[1, 0, 1]] * 7, opacity=[0.5] * 7, rgb=[[1, 1, 1]] * 7,
                depth=[1.0] * 7)
    sc = scene_of(32, 32, **base)
    sc.depth[1] = 0.0                 # not in front
    sc.conic[2] = [1.0, 2.0, 1.0]     # not positive definite
    sc.opacity[3] = 0.5 / 255.0       # can never reach 1/255
    sc.mean2d[4, 0] = np.nan          # non-finite
    sc.conic[5] = [-1.0, 0.0, -1.0]   # negative definite
    sc.rgb[6, 1] = np.inf
    _, vals, count, culled = oracle.bin_tiles(sc)
    assert culled == 6 and set(vals.tolist()) == {0}


def test_translation_by_one_tile():
    """Moving every splat 16 px right moves each interior splat's pairs one
    tile right and the image 16 px right."""
    sc = synth.make_scene(1, seed=11, n=60, W=128, H=64)
    sc.mean2d[:, 0] = 20 + (sc.mean2d[:, 0] % 60)
    sc.mean2d[:] = np.round(sc.mean2d * 1024) / 1024   # mean and mean + 16 exact in float32
    sc2 = synth.Scene(**{**sc.__dict__})
    sc2.mean2d = sc.mean2d.copy()
    sc2.mean2d[:, 0] += 16
    k1, v1, _, _ = oracle.bin_tiles(sc)
    k2, v2, _, _ = oracle.bin_tiles(sc2)
    p1 = sorted(zip(v1.tolist(), ((k1 >> np.uint64(32)) + np.uint64(1)).tolist()))
    p2 = sorted(zip(v2.tolist(), (k2 >> np.uint64(32)).tolist()))
    assert p1 == p2
    _, f1 = render(sc)
    _, f2 = render(sc2)
    assert np.array_equal(f1["image"][:, :, 0:100], f2["image"][:, :, 16:116])


# ---------------------------------------------------------------- sort / offsets

def test_sort_and_offsets_match_library():
    rng = np.random.default_rng(5)
    n = 5000
    tiles = rng.integers(0, 37, n).astype(np.uint64)
    dep = rng.choice(np.float32([1.0, 1.5, 2.25, 7.0, 9.5]), n)  # many exact ties
    keys = (tiles << np.uint64(32)) | dep.view(np.uint32).astype(np.uint64)
    vals = rng.permutation(n).astype(np.uint32)
    sk, sv = oracle.sort_pairs(keys, vals)
    ref = sorted(zip(keys.tolist(), vals.tolist()))
    assert list(zip(sk.tolist(), sv.tolist())) == ref
    offs = oracle.offsets(sk, 40)
    assert np.array_equal(offs, np.searchsorted((sk >> np.uint64(32)).astype(np.int64),
                                                np.arange(41), side="left").astype(np.uint32))
    # depth bits order = depth order for positive floats
    d = np.sort(rng.uniform(0.001, 1e4, 1000).astype(np.float32))
    assert np.all(np.diff(d.view(np.uint32).astype(np.int64)) >= 0)


# ---------------------------------------------------------------- forward closed forms

def test_single_isotropic_splat_closed_form():
    s, o, col = 2.5, 0.8, (0.2, 0.5, 0.9)
    sc = scene_of(48, 48, [[20.5, 17.5]], [[1 / s**2, 0, 1 / s**2]], [o], [col], [3.0])
    _, f = render(sc)
    ys, xs = np.mgrid[0:48, 0:48]
    r2 = (xs + 0.5 - 20.5) ** 2 + (ys + 0.5 - 17.5) ** 2
    a32 = float(np.float32(1 / s**2))
    al = np.minimum(0.99, float(np.float32(o)) * np.exp(-0.5 * r2 * a32))
    al = np.where(al >= ALPHA_MIN, al, 0.0)
    for ch in range(3):
        np.testing.assert_allclose(f["image"][ch], np.float32(col[ch]) * al, atol=1e-12)
    np.testing.assert_allclose(f["T_final"], 1 - al, atol=1e-12)
    assert f["last"][17, 20] == 1 and f["image"][0, 17, 20] == pytest.approx(np.float32(0.2) * np.float32(0.8))
    assert np.array_equal(f["last"] == 1, al > 0)
    assert np.all(f["median"][al > 0] == 3.0)


def test_two_splats_front_to_back_by_depth():
    a1, a2 = 0.6, 0.7
    c1, c2 = (1.0, 0.0, 0.0), (0.0, 1.0, 0.0)
    for d1, d2 in ((1.0, 2.0), (2.0, 1.0)):
        sc = scene_of(16, 16, [[8.5, 8.5]] * 2, [[4, 0, 4]] * 2, [a1, a2], [c1, c2], [d1, d2],
                      bg=(0.1, 0.2, 0.3))
        _, f = render(sc)
        p = (8, 8)
        A1, A2 = float(np.float32(a1)), float(np.float32(a2))
        if d1 < d2:
            C = np.array(c1) * A1 + np.array(c2) * A2 * (1 - A1)
        else:
            C = np.array(c2) * A2 + np.array(c1) * A1 * (1 - A2)
        T = (1 - A1) * (1 - A2)
        np.testing.assert_allclose(f["image"][:, p[1], p[0]], C + T * np.float32([0.1, 0.2, 0.3]),
                                   atol=1e-12)
        assert f["T_final"][p[1], p[0]] == pytest.approx(T, abs=1e-15)
        assert f["last"][p[1], p[0]] == 2


def test_termination_rule():
    """alpha 0.95 repeated: T = 0.05, 0.0025, 1.25e-4 after 3 blends; the 4th
    would give 6.25e-6 < 1e-4, so exactly 3 blend."""
    n = 6
    sc = scene_of(16, 16, [[8.5, 8.5]] * n, [[50, 0, 50]] * n, [0.95] * n, [[1, 1, 1]] * n,
                  np.arange(1, n + 1))
    _, f = render(sc)
    A = float(np.float32(0.95))
    assert f["last"][8, 8] == 3
    assert f["T_final"][8, 8] == pytest.approx((1 - A) ** 3, rel=1e-14)
    assert f["image"][0, 8, 8] == pytest.approx(1 - (1 - A) ** 3, rel=1e-14)


def test_median_depth_closed_form():
    sc = scene_of(16, 16, [[8.5, 8.5]] * 3, [[50, 0, 50]] * 3, [0.3, 0.5, 0.4], [[1, 1, 1]] * 3,
                  [1.0, 2.0, 3.0])
    _, f = render(sc)
    assert f["median"][8, 8] == 2.0      # T before: 1, 0.7, 0.35
    sc.opacity[:] = np.float32([0.7, 0.5, 0.4])
    _, f = render(sc)
    assert f["median"][8, 8] == 1.0      # T before: 1, 0.3
    assert f["median"][0, 0] == 0.0      # nothing blended


def test_invariants_white_splats():
    sc = synth.make_scene(1, seed=2)
    sc.rgb[:] = 1.0
    sc.bg = np.ones(3, np.float32)
    _, f = render(sc)
    np.testing.assert_allclose(f["image"], 1.0, atol=1e-13)
    sc.bg = np.zeros(3, np.float32)
    _, f = render(sc)
    for ch in range(3):
        np.testing.assert_allclose(f["image"][ch], 1.0 - f["T_final"], atol=1e-13)


@pytest.mark.parametrize("wl,n,W,H", [(1, 256, 64, 64), (2, 5207, 256, 256), (3, 3000, 250, 170)])
def test_tiled_equals_brute_force_over_all_splats(wl, n, W, H):
    """Per pixel, compositing every valid splat in (depth, index) order,
    ignoring tiles, gives the same doubles as the tiled lists."""
    sc = synth.make_scene(wl, seed=1, n=n, W=W, H=H)
    tl, f = render(sc)
    valid = np.array([oracle.splat_rect(sc, i)[0] >= 0 for i in range(sc.n)])
    idx = np.nonzero(valid)[0]
    order = idx[np.lexsort((idx, sc.depth[idx]))].astype(np.uint32)
    tx, ty = oracle.tiles_xy(W, H)
    vals = np.tile(order, tx * ty)
    offs = (np.arange(tx * ty + 1) * order.size).astype(np.uint32)
    b = oracle.forward(sc, vals, offs)
    for k in ("image", "T_final", "last", "median", "dist"):
        if k == "last":   # positions differ (whole list vs tile list); compare the splat
            lt = np.zeros_like(f[k], np.int64) - 1
            lb = np.zeros_like(b[k], np.int64) - 1
            for y in range(H):
                for x in range(W):
                    t = (y // 16) * tx + x // 16
                    if f[k][y, x]:
                        lt[y, x] = tl["vals"][tl["offs"][t] + f[k][y, x] - 1]
                    if b[k][y, x]:
                        lb[y, x] = order[b[k][y, x] - 1]
            assert np.array_equal(lt, lb)
        else:
            assert np.array_equal(f[k], b[k]), k


def test_weight_statistics_single_splat_closed_form():
    """max blend weight = alpha at the pixel centre nearest the mean, count =
    pixels with alpha >= 1/255 (one splat, T = 1 everywhere)."""
    s, o = 2.0, 0.6
    sc = scene_of(40, 40, [[19.3, 21.8]], [[1 / s**2, 0, 1 / s**2]], [o], [[1, 1, 1]], [2.0])
    _, f = render(sc)
    ys, xs = np.mgrid[0:40, 0:40]
    a32 = float(np.float32(1 / s**2))
    r2 = (xs + 0.5 - float(np.float32(19.3))) ** 2 + (ys + 0.5 - float(np.float32(21.8))) ** 2
    al = float(np.float32(o)) * np.exp(-0.5 * r2 * a32)
    assert f["max_w"][0] == pytest.approx(al.max(), rel=1e-14)
    assert f["count"][0] == int((al >= ALPHA_MIN).sum())


def test_weight_statistics_consistent_with_backward():
    """count >= 1 and max_w > 0 exactly for splats with a positive accumulated
    weight, and max_w <= accum <= count * max_w."""
    sc = synth.make_scene(2, seed=5, n=1500, W=128, H=96)
    tl, f = render(sc)
    acc = oracle.backward(sc, tl["vals"], tl["offs"])["grads"]["accum"]
    pos = acc > 0
    assert np.array_equal(pos, f["count"] > 0) and np.array_equal(pos, f["max_w"] > 0)
    assert np.all(f["max_w"][pos] <= acc[pos] * (1 + 1e-12))
    assert np.all(acc[pos] <= f["count"][pos] * f["max_w"][pos] * (1 + 1e-12))


# ---------------------------------------------------------------- knife edges

def test_knife_edge_pixel_has_alternative():
    """A splat tuned so that alpha is 1/255 within 1e-9 at one pixel centre:
    the oracle flags that pixel and reports the outcome with the other decision."""
    s = 2.0
    o = np.float32(0.5)
    # distance where o exp(-r^2 / (2 s^2)) = 1/255 exactly
    r = s * math.sqrt(2 * math.log(255 * float(o)))
    sc = scene_of(32, 32, [[0.5 + r, 10.5]], [[1 / s**2, 0, 1 / s**2]], [o], [[1, 1, 1]], [1.0])
    _, f = render(sc)
    assert f["n_amb"][10, 0] >= 1
    alts = f["alts"]
    assert np.any((alts["pixel"] == 10 * 32 + 0) & (alts["kind"] == oracle.AMB_ALPHA))
    a = alts[(alts["pixel"] == 10 * 32 + 0) & (alts["kind"] == oracle.AMB_ALPHA)][0]
    assert {int(a["last"]), int(f["last"][10, 0])} == {0, 1}
    assert (f["n_amb"] > 0).sum() <= 3


# ---------------------------------------------------------------- backward

def _loss(sc, tl, params, bg, gD=None):
    f = oracle.forward(sc, tl["vals"], tl["offs"], params=params, bg=bg)
    L = float(np.sum(f["image"] * sc.dL_dimage.astype(np.float64)))
    if gD is not None:
        L += float(np.sum(f["dist"] * gD))
    return L


FIELDS = [("mean2d", "dmean2d", 2), ("conic", "dconic", 3), ("opacity", "dopacity", 1),
          ("rgb", "drgb", 3)]


@pytest.mark.parametrize("seed,clamp,dist", [(0, False, False), (1, False, False),
                                             (2, True, False), (3, False, True),
                                             (4, True, True)])
def test_backward_matches_central_finite_differences(seed, clamp, dist):
    rng = np.random.default_rng(seed)
    n, W, H = 12, 32, 32
    th = rng.uniform(0, np.pi, n)
    s1, s2 = np.exp(rng.uniform(0, 1.4, n)), np.exp(rng.uniform(0, 1.4, n))
    conic = synth.conic_from_scales(th, s1, s2)
    op = rng.uniform(0.2, 0.9, n)
    if clamp:
        op[:4] = 1.0   # alpha clamps to 0.99 near these centres
    sc = scene_of(W, H, rng.uniform(5, 27, (n, 2)), conic, op, rng.uniform(0, 1, (n, 3)),
                  rng.permutation(n) + 1.0, dL=rng.normal(0, 1, (3, H, W)), bg=(0.2, 0.3, 0.4))
    tl = oracle.tile_lists(sc)
    bgd = sc.bg.astype(np.float64)
    base = {k: getattr(sc, k).astype(np.float64) for k in ("mean2d", "conic", "opacity", "rgb", "depth")}
    gD = rng.normal(0, 0.05, (H, W)) if dist else None
    an = oracle.backward(sc, tl["vals"], tl["offs"], dL_ddist=gD)["grads"]
    checked = 0
    fields = FIELDS + ([("depth", "ddepth", 1)] if dist else [])
    for name, gname, width in fields:
        ref = np.abs(an[gname]).max()
        for i in range(n):
            for c in range(width):
                def fd(h):
                    p1 = {k: v.copy() for k, v in base.items()}
                    p2 = {k: v.copy() for k, v in base.items()}
                    p1[name].reshape(n, -1)[i, c] += h
                    p2[name].reshape(n, -1)[i, c] -= h
                    return (_loss(sc, tl, p1, bgd, gD) - _loss(sc, tl, p2, bgd, gD)) / (2 * h)
                x = abs(base[name].reshape(n, -1)[i, c])
                h = 1e-5 * max(1.0, x)
                f1, f2 = fd(h), fd(h / 2)
                if abs(f1 - f2) > 1e-4 * max(abs(f1), 1e-3 * ref):
                    continue   # a decision flips within +-h: not differentiable here
                g = an[gname].reshape(n, -1)[i, c]
                assert abs(f2 - g) <= 2e-6 * max(abs(g), 1e-2 * ref), (name, i, c, f2, g)
                checked += 1
    assert checked >= 0.9 * n * (10 if dist else 9)


def test_distortion_two_splats_closed_form():
    a1, a2 = 0.6, 0.7
    for d1, d2 in ((1.0, 4.0), (4.0, 1.0)):
        sc = scene_of(16, 16, [[8.5, 8.5]] * 2, [[4, 0, 4]] * 2, [a1, a2], [[1, 1, 1]] * 2,
                      [d1, d2])
        _, f = render(sc)
        A1, A2 = float(np.float32(a1)), float(np.float32(a2))
        wf, wb = (A1, A2 * (1 - A1)) if d1 < d2 else (A2, A1 * (1 - A2))
        assert f["dist"][8, 8] == pytest.approx(wf * wb * 9.0, rel=1e-14)
    sc = scene_of(16, 16, [[8.5, 8.5]] * 3, [[4, 0, 4]] * 3, [0.5, 0.5, 0.5], [[1, 1, 1]] * 3,
                  [1.0, 2.0, 5.0])
    _, f = render(sc)
    w = [0.5, 0.25, 0.125]
    ref = w[0] * w[1] * 1 + w[0] * w[2] * 16 + w[1] * w[2] * 9
    assert f["dist"][8, 8] == pytest.approx(ref, rel=1e-14)


def test_distortion_invariants():
    sc = synth.make_scene(2, seed=4, n=600, W=64, H=48)
    _, f = render(sc)
    assert np.all(f["dist"] >= 0) and f["dist"].max() > 0
    one = synth.subset(sc, np.array([5]))
    assert not render(one)[1]["dist"].any()                    # one splat: no pair
    flat = synth.subset(sc, np.arange(sc.n))
    flat.depth[:] = np.float32(3.0)
    assert not render(flat)[1]["dist"].any()                   # equal depths
    dbl = synth.subset(sc, np.arange(sc.n))
    dbl.depth *= np.float32(2.0)                               # exact; same order
    np.testing.assert_allclose(render(dbl)[1]["dist"], 4.0 * f["dist"], rtol=1e-12, atol=0)


def test_accum_weight_equals_red_gradient_under_unit_red_loss():
    sc = synth.make_scene(1, seed=4)
    tl = oracle.tile_lists(sc)
    g = np.zeros((3, sc.H, sc.W))
    g[0] = 1.0
    b = oracle.backward(sc, tl["vals"], tl["offs"], dL_dimage=g)["grads"]
    assert np.array_equal(b["drgb"][:, 0], b["accum"])
    assert np.all(b["drgb"][:, 1:] == 0)


def test_accum_weight_single_splat_closed_form():
    s, o = 3.0, 0.7
    sc = scene_of(40, 40, [[19.3, 21.8]], [[1 / s**2, 0, 1 / s**2]], [o], [[1, 1, 1]], [2.0])
    tl = oracle.tile_lists(sc)
    b = oracle.backward(sc, tl["vals"], tl["offs"])["grads"]
    ys, xs = np.mgrid[0:40, 0:40]
    r2 = (xs + 0.5 - float(np.float32(19.3))) ** 2 + (ys + 0.5 - float(np.float32(21.8))) ** 2
    al = float(np.float32(o)) * np.exp(-0.5 * r2 * float(np.float32(1 / s**2)))
    assert b["accum"][0] == pytest.approx(al[al >= ALPHA_MIN].sum(), rel=1e-13)


def test_backward_tile_mask_is_additive():
    """Gradients from disjoint tile masks sum to the whole-image gradient."""
    sc = synth.make_scene(2, seed=9, n=800, W=96, H=80)
    tl = oracle.tile_lists(sc)
    tx, ty = oracle.tiles_xy(sc.W, sc.H)
    m1 = (np.arange(tx * ty) % 3 == 0).astype(np.uint8)
    full = oracle.backward(sc, tl["vals"], tl["offs"])["grads"]
    g1 = oracle.backward(sc, tl["vals"], tl["offs"], tile_mask=m1)["grads"]
    g2 = oracle.backward(sc, tl["vals"], tl["offs"], tile_mask=1 - m1)["grads"]
    for k in full:
        np.testing.assert_allclose(g1[k] + g2[k], full[k], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- planted mistakes

MUTATIONS = [
    ("rx uses a", "const float rx = sqrtf(k * c / det);", "const float rx = sqrtf(k * a / det);"),
    ("pixel corner not centre", "run_pixel(s, list, len, x + 0.5, y + 0.5, -1, 0, &r);\n                    if (out->image)",
     "run_pixel(s, list, len, x + 0.0, y + 0.5, -1, 0, &r);\n                    if (out->image)"),
    ("b term sign", "const double sigma = 0.5 * (a * dx * dx + c * dy * dy) + b * dx * dy;",
     "const double sigma = 0.5 * (a * dx * dx + c * dy * dy) - b * dx * dy;"),
    ("termination after blend", "if (stop)\n            break;", "if (stop && 0)\n            break;"),
    ("dropped bg in dL/dalpha", "(S[ch] + r->T * bg[ch])", "(S[ch])"),
    ("dmean_y uses a", "o[F_MY] = dL_dsigma * -(b * dx + c * dy);", "o[F_MY] = dL_dsigma * -(b * dx + a * dy);"),
    ("db halved", "o[F_B] = dL_dsigma * dx * dy;", "o[F_B] = dL_dsigma * 0.5 * dx * dy;"),
    ("dopacity without G", "o[F_O] = dL_dalpha * e->G;", "o[F_O] = dL_dalpha;"),
    ("sort descending", "return a->key < b->key ? -1 : 1;", "return a->key < b->key ? 1 : -1;"),
    ("median uses first", "if (med)\n            r->median", "if (med && r->median == 0.0)\n            r->median"),
    ("k margin dropped", "k = k * K_REL + K_ABS;", "k = k * 0.9f;"),
    ("max weight over alpha", "const double w = r.rec[k].alpha * r.rec[k].T;",
     "const double w = r.rec[k].alpha;"),
    ("count of evaluated splats", "out->count[i] += 1;", "out->count[i] += 2;"),
    ("distortion |dz|", "D += wi * wj * dz * dz;", "D += wi * wj * fabs(dz);"),
    ("distortion without the later splats' term",
     "dL_dalpha += gD * (E * e->T - SE / (1.0 - e->alpha));", "dL_dalpha += gD * (E * e->T);"),
    ("ddepth halved", "dz_sum += 2.0 * w * wj * dz;", "dz_sum += w * wj * dz;"),
    ("suffix sum without w", "SE += w * E;", "SE += E;"),
]


def _run_mutant(tmp_dir, idx, old, new):
    """Build oracle.c with one planted mistake and run the fast pins on it;
    returns the pin run's exit code (0: every pin passed)."""
    here = os.path.dirname(oracle.__file__)
    src = open(os.path.join(here, "oracle.c")).read()
    if src.count(old) != 1:
        return "pattern"
    d = os.path.join(tmp_dir, "m%02d" % idx)
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
    """All planted mistakes, run concurrently (independent subprocesses)."""
    import concurrent.futures as cf
    tmp = str(tmp_path_factory.mktemp("mutants"))
    workers = max(1, min(len(MUTATIONS), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        futs = [ex.submit(_run_mutant, tmp, i, old, new)
                for i, (_, old, new) in enumerate(MUTATIONS)]
        return [f.result() for f in futs]


@pytest.mark.slow
@pytest.mark.parametrize("k", range(len(MUTATIONS)), ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(mutant_results, k):
    label = MUTATIONS[k][0]
    assert mutant_results[k] != "pattern", "mutation '%s' does not match oracle.c" % label
    assert mutant_results[k] != 0, "planted mistake '%s' passed every pin" % label
