"""Parity of the CUDA path (through the C ABI) against the CPU oracle.

Tolerances (the rasterizer's stated bar):
  * pairs (as a multiset), sorted keys/values, tile offsets: bit-exact;
  * image, T_final: 1e-5 absolute; last_contrib and median depth: exact;
  * depth distortion: max(1e-5, e_D), e_D the oracle's bound on a float32
    evaluation by running totals (the totals' terms z'^2 A, z' D1, D2 are
    large next to their difference when depths are far apart); dL/ddepth
    under the gradient bar below;
  * per-splat max blend weight: 1e-5 absolute; blending-pixel count: exact
    (splats blended at a knife-edge pixel in some outcome are skipped);
  * gradients: max(1e-4, 1e-3 * max|field|) per element, field = one of
    dmean2d, dconic, dopacity, drgb;
  * accumulated weight: max(1e-5, e) + 2^-23 |w|, e = the oracle's bound on the
    error of a float32 evaluation of the sum (1e-5 alone is below one float32
    ulp for sums above 128), the last term the output's own rounding.
A knife-edge pixel (a float32 decision within rounding of its threshold)
must equal the oracle's normal outcome or one of its alternatives; each
gradient element's tolerance grows by the oracle's slack, the sum over knife
edges of |alternative - normal| contribution.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import gaussian_splatting_differentiable_gb300 as ss

GRAD_FIELDS = ("dmean2d", "dconic", "dopacity", "drgb")
DIST_FIELD = "ddepth"


def flags_of(scene) -> int:
    return (ss.SS_ACCUM_WEIGHT if scene.accum_weight else 0) | \
        (ss.SS_MEDIAN_DEPTH if scene.median_depth else 0) | \
        (ss.SS_WEIGHT_STATS if getattr(scene, "weight_stats", False) else 0) | \
        (ss.SS_DISTORTION if getattr(scene, "distortion", False) else 0)


def run_gpu_graph(scene):
    """The step as bench.py times it: pair buffers of 2.5 n, one synchronous
    step to size them, then the CUDA graph of bin -> sort on the device-side
    pair count -> forward -> backward, replayed twice; numpy copies of the
    outputs of the last replay (the binned, unsorted pairs are not kept by
    this path, so the multiset check uses the sorted ones)."""
    dev = torch.device("cuda")
    sp = ss.Splats.from_numpy(scene, dev)
    flags = flags_of(scene)
    r = ss.Rasterizer(scene.W, scene.H, scene.n, int(2.5 * scene.n), flags, bg=scene.bg,
                      device=dev)
    dL = torch.from_numpy(scene.dL_dimage).to(dev).contiguous()
    dLd = (torch.from_numpy(scene.dL_ddist).to(dev).contiguous()
           if flags & ss.SS_DISTORTION else None)
    r.step(sp, dL, dL_ddist=dLd)
    g = r.capture(sp, dL, dL_ddist=dLd)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    r.check()
    st, pairs, culled = ss.ss_pair_count(r.counters, r.capacity)
    assert st == ss.SS_OK
    out = {"count": pairs, "culled": culled, "sort_status": ss.ss_sort_status(r.workspace)}
    out["keys"] = r.keys[:pairs].cpu().numpy().view(np.uint64).copy()
    out["vals"] = r.vals[:pairs].cpu().numpy().view(np.uint32).copy()
    out["keys_binned"], out["vals_binned"] = out["keys"], out["vals"]
    out["offs"] = r.tile_offsets.cpu().numpy().view(np.uint32).copy()
    out["image"] = r.image.cpu().numpy()
    out["T_final"] = r.T_final.cpu().numpy()
    out["last"] = r.last_contrib.cpu().numpy().view(np.uint32)
    out["median"] = r.median_depth.cpu().numpy() if r.median_depth is not None else None
    out["dist"] = r.distortion.cpu().numpy() if r.distortion is not None else None
    for k in GRAD_FIELDS + (DIST_FIELD,):
        out[k] = r.grads[k].cpu().numpy() if k in r.grads else None
    out["accum"] = r.accum_weight.cpu().numpy() if r.accum_weight is not None else None
    out["max_w"] = r.max_weight.cpu().numpy() if r.max_weight is not None else None
    out["bcount"] = (r.blend_count.cpu().numpy().view(np.uint32)
                     if r.blend_count is not None else None)
    return out


def run_gpu(scene, capacity=None, stream=None):
    """Whole path through the C ABI; returns numpy copies of every stage."""
    dev = torch.device("cuda")
    sp = ss.Splats.from_numpy(scene, dev)
    flags = flags_of(scene)
    cap = capacity if capacity is not None else max(64, 4 * scene.n)
    r = ss.Rasterizer(scene.W, scene.H, scene.n, cap, flags, bg=scene.bg, device=dev)
    ss.ss_bin_tiles(sp, scene.W, scene.H, r.keys, r.vals, r.capacity, r.counters, r.records, stream)
    st, pairs, culled = ss.ss_pair_count(r.counters, r.capacity, stream)
    if st != ss.SS_OK:
        r._alloc_pairs(pairs + 16)
        ss.ss_bin_tiles(sp, scene.W, scene.H, r.keys, r.vals, r.capacity, r.counters, r.records,
                        stream)
        st, pairs, culled = ss.ss_pair_count(r.counters, r.capacity, stream)
        assert st == ss.SS_OK
    out = {"count": pairs, "culled": culled,
           "keys_binned": r.keys[:pairs].cpu().numpy().view(np.uint64).copy(),
           "vals_binned": r.vals[:pairs].cpu().numpy().view(np.uint32).copy()}
    r.n_pairs = pairs
    ss.ss_sort_pairs(r.keys, r.vals, pairs, scene.W, scene.H, r.tile_offsets, r.workspace, stream)
    out["sort_status"] = ss.ss_sort_status(r.workspace, stream)
    out["keys"] = r.keys[:pairs].cpu().numpy().view(np.uint64).copy()
    out["vals"] = r.vals[:pairs].cpu().numpy().view(np.uint32).copy()
    out["offs"] = r.tile_offsets.cpu().numpy().view(np.uint32).copy()
    r.forward(sp, stream)
    dL = torch.from_numpy(scene.dL_dimage).to(dev).contiguous()
    dLd = (torch.from_numpy(scene.dL_ddist).to(dev).contiguous()
           if flags & ss.SS_DISTORTION else None)
    r.backward(sp, dL, stream, dLd)
    torch.cuda.synchronize()
    out["image"] = r.image.cpu().numpy()
    out["T_final"] = r.T_final.cpu().numpy()
    out["last"] = r.last_contrib.cpu().numpy().view(np.uint32)
    out["median"] = r.median_depth.cpu().numpy() if r.median_depth is not None else None
    out["dist"] = r.distortion.cpu().numpy() if r.distortion is not None else None
    for k in GRAD_FIELDS + (DIST_FIELD,):
        out[k] = r.grads[k].cpu().numpy() if k in r.grads else None
    out["accum"] = r.accum_weight.cpu().numpy() if r.accum_weight is not None else None
    out["max_w"] = r.max_weight.cpu().numpy() if r.max_weight is not None else None
    out["bcount"] = (r.blend_count.cpu().numpy().view(np.uint32)
                     if r.blend_count is not None else None)
    return out


def _outputs(r, out):
    """numpy copies of a Rasterizer's outputs into out."""
    torch.cuda.synchronize()
    out["image"] = r.image.cpu().numpy()
    out["T_final"] = r.T_final.cpu().numpy()
    out["last"] = r.last_contrib.cpu().numpy().view(np.uint32)
    out["median"] = r.median_depth.cpu().numpy() if r.median_depth is not None else None
    out["dist"] = r.distortion.cpu().numpy() if r.distortion is not None else None
    for k in GRAD_FIELDS + (DIST_FIELD,):
        out[k] = r.grads[k].cpu().numpy() if k in r.grads else None
    out["accum"] = r.accum_weight.cpu().numpy() if r.accum_weight is not None else None
    out["max_w"] = r.max_weight.cpu().numpy() if r.max_weight is not None else None
    out["bcount"] = (r.blend_count.cpu().numpy().view(np.uint32)
                     if r.blend_count is not None else None)
    return out


def run_gpu_splats(scene):
    """bin -> sort -> ss_raster_fwd -> ss_raster_bwd, the entry points that
    take the splats themselves: no records and no blend masks are passed
    (the forward computes each batch's records, the backward rebuilds the
    records and re-evaluates the blend decisions in its workspace).  The
    optional outputs these calls have: accumulated weight, median depth."""
    dev = torch.device("cuda")
    sp = ss.Splats.from_numpy(scene, dev)
    flags = flags_of(scene) & (ss.SS_ACCUM_WEIGHT | ss.SS_MEDIAN_DEPTH)
    r = ss.Rasterizer(scene.W, scene.H, scene.n, max(64, 4 * scene.n), flags, bg=scene.bg,
                      device=dev)
    pairs = r.bin_and_sort(sp)
    out = {"count": pairs, "culled": r.culled}
    out["keys"] = r.keys[:pairs].cpu().numpy().view(np.uint64).copy()
    out["vals"] = r.vals[:pairs].cpu().numpy().view(np.uint32).copy()
    out["keys_binned"], out["vals_binned"] = out["keys"], out["vals"]
    out["offs"] = r.tile_offsets.cpu().numpy().view(np.uint32).copy()
    r.image.fill_(float("nan"))
    ss.ss_raster_fwd(sp, r.vals, r.tile_offsets, scene.W, scene.H, r.bg, flags, r.image,
                     r.T_final, r.last_contrib, r.median_depth)
    dL = torch.from_numpy(scene.dL_dimage).to(dev).contiguous()
    for v in r.grads.values():
        v.fill_(float("nan"))
    ss.ss_raster_bwd(sp, r.vals, r.tile_offsets, scene.W, scene.H, r.bg, flags, r.T_final,
                     r.last_contrib, dL, r.grads, r.accum_weight, r.workspace)
    out["sort_status"] = ss.ss_sort_status(r.workspace)
    return _outputs(r, out)


def run_gpu_nomask(scene):
    """The records path with the backward given no blend masks
    (ss_raster_bwd_records re-evaluates the decisions into its workspace)."""
    dev = torch.device("cuda")
    sp = ss.Splats.from_numpy(scene, dev)
    flags = flags_of(scene)
    r = ss.Rasterizer(scene.W, scene.H, scene.n, max(64, 4 * scene.n), flags, bg=scene.bg,
                      device=dev)
    pairs = r.bin_and_sort(sp)
    out = {"count": pairs, "culled": r.culled}
    out["keys"] = r.keys[:pairs].cpu().numpy().view(np.uint64).copy()
    out["vals"] = r.vals[:pairs].cpu().numpy().view(np.uint32).copy()
    out["keys_binned"], out["vals_binned"] = out["keys"], out["vals"]
    out["offs"] = r.tile_offsets.cpu().numpy().view(np.uint32).copy()
    r.forward(sp)
    r.blend_masks.fill_(-1)              # the backward must not read them
    dL = torch.from_numpy(scene.dL_dimage).to(dev).contiguous()
    dLd = (torch.from_numpy(scene.dL_ddist).to(dev).contiguous()
           if flags & ss.SS_DISTORTION else None)
    ss.ss_raster_bwd_records(r.records, r.n, r.vals, r.tile_offsets, r.n_pairs, scene.W, scene.H,
                             r.bg, flags | ss.SS_RECORDS_CLEARED, r.T_final, r.last_contrib, None,
                             dL, r.grads, r.accum_weight, r.workspace, None, r.dist_totals, dLd)
    out["sort_status"] = ss.ss_sort_status(r.workspace)
    return _outputs(r, out)


def _pairs_sorted(keys, vals):
    o = np.lexsort((vals, keys))
    return keys[o], vals[o]


def check_pairs(scene, gpu, orc=None):
    orc = orc or oracle.tile_lists(scene)
    assert gpu["sort_status"] == ss.SS_OK
    assert gpu["count"] == orc["count"], (gpu["count"], orc["count"])
    assert gpu["culled"] == orc["culled"]
    gk, gv = _pairs_sorted(gpu["keys_binned"], gpu["vals_binned"])
    assert np.array_equal(gk, orc["keys"]) and np.array_equal(gv, orc["vals"]), "binned multiset"
    assert np.array_equal(gpu["keys"], orc["keys"]), "sorted keys"
    assert np.array_equal(gpu["vals"], orc["vals"]), "sorted values"
    assert np.array_equal(gpu["offs"], orc["offs"]), "tile offsets"
    return orc


# Largest fraction of compared pixels that may be knife edges: 1e-4 on the
# smaller workloads; the 2M-splat ones blend ~70 splats a pixel, and the
# sound (worst-case) bound on the float32 transmittance grows with the chain,
# so more termination decisions fall inside it (measured 4.1e-4 on the
# 1237x822 scene).
KNIFE_EDGE_CAP = 1e-4
KNIFE_EDGE_CAP_DENSE = 5e-4


def relevant_knife_edges(scene, ofw):
    """Pixels with a knife-edge decision that can change a compared output:
    the alpha floor, the alpha cap and the termination always; the T = 0.5
    decision only when the median depth is an output.  A pixel with more
    flagged decisions than the oracle listed alternatives for counts as
    flagged."""
    H, W = scene.H, scene.W
    alts = ofw["alts"]
    kinds = [oracle.AMB_ALPHA, oracle.AMB_TERM, oracle.AMB_CLAMP]
    if scene.median_depth:
        kinds.append(oracle.AMB_MEDIAN)
    amb = np.zeros(H * W, bool)
    amb[alts["pixel"][np.isin(alts["kind"], kinds)]] = True
    listed = np.bincount(alts["pixel"], minlength=H * W)
    amb |= ofw["n_amb"].reshape(-1).astype(np.int64) > listed
    return amb.reshape(H, W)


def check_forward(scene, gpu, ofw, pixel_mask=None, atol=1e-5, knife_cap=None):
    """Compare per pixel; returns dict of counts.  knife_cap: if given, the
    knife-edge pixels (relevant_knife_edges) must be fewer than this
    fraction of the compared pixels."""
    H, W = scene.H, scene.W
    sel = np.ones((H, W), bool) if pixel_mask is None else pixel_mask
    flagged = relevant_knife_edges(scene, ofw)
    clean = sel & ~flagged
    img_err = np.abs(gpu["image"] - ofw["image"]).max(axis=0)
    T_err = np.abs(gpu["T_final"] - ofw["T_final"])
    bad = clean & ((img_err > atol) | (T_err > atol) | (gpu["last"] != ofw["last"]))
    if gpu["median"] is not None:
        bad |= clean & (gpu["median"] != ofw["median"].astype(np.float32))
    dist_tol = np.maximum(atol, ofw["dist_err"])
    if gpu.get("dist") is not None:
        dist_err = np.abs(gpu["dist"] - ofw["dist"])
        bad_d = clean & (dist_err > dist_tol)
        assert not bad_d.any(), "distortion: %d pixels off; worst err %.3g (tol %.3g)" % (
            bad_d.sum(), dist_err[bad_d].max(), dist_tol[bad_d][np.argmax(dist_err[bad_d])])
    assert not bad.any(), _describe_bad(bad, gpu, ofw, img_err, T_err)
    # knife edges: the GPU must take the normal outcome or one alternative
    amb = np.argwhere(sel & flagged)
    if knife_cap is not None:
        assert len(amb) < knife_cap * max(int(sel.sum()), 1), (
            "%d knife-edge pixels of %d compared: not below %.0e" % (len(amb), sel.sum(),
                                                                      knife_cap))
    alts = ofw["alts"]
    unmatched = 0
    for (y, x) in amb:
        p = y * W + x
        cands = [(ofw["image"][:, y, x], ofw["T_final"][y, x], ofw["last"][y, x],
                  ofw["median"][y, x], ofw["dist"][y, x])]
        for a in alts[alts["pixel"] == p]:
            cands.append((a["image"], a["T_final"], a["last"], a["median"], a["dist"]))
        ok = False
        for im, T, last, med, dd in cands:
            if (np.abs(gpu["image"][:, y, x] - im).max() <= atol and abs(gpu["T_final"][y, x] - T) <= atol
                    and gpu["last"][y, x] == last
                    and (gpu["median"] is None or gpu["median"][y, x] == np.float32(med))
                    and (gpu.get("dist") is None
                         or abs(gpu["dist"][y, x] - dd) <= 2 * dist_tol[y, x])):
                ok = True
                break
        unmatched += not ok
    assert unmatched == 0, "%d knife-edge pixels match no oracle outcome" % unmatched
    return {"pixels": int(sel.sum()), "knife_edge": int(len(amb)),
            "max_img_err": float(img_err[clean].max()) if clean.any() else 0.0}


def check_weight_stats(scene, gpu, ofw, splat_mask=None, atol=1e-5):
    """Per-splat max blend weight and blending-pixel count; ofw must cover
    every tile of the selected splats."""
    if gpu["max_w"] is None:
        return None
    sel = np.ones(scene.n, bool) if splat_mask is None else splat_mask
    clean = sel & (ofw["splat_amb"] == 0)
    err = np.abs(gpu["max_w"].astype(np.float64) - ofw["max_w"])
    bad = clean & (err > atol)
    assert not bad.any(), "max weight: %d splats off; worst %.3g" % (bad.sum(), err[bad].max())
    badc = clean & (gpu["bcount"] != ofw["count"])
    assert not badc.any(), "blend count: %d splats off; first %d gpu %d oracle %d" % (
        badc.sum(), np.argmax(badc), gpu["bcount"][np.argmax(badc)],
        ofw["count"][np.argmax(badc)])
    return {"splats": int(clean.sum()), "knife_edge_splats": int((sel & ~clean).sum()),
            "max_w_err": float(err[clean].max(initial=0.0)),
            "blended": int((clean & (ofw["count"] > 0)).sum())}


def _describe_bad(bad, gpu, ofw, img_err, T_err):
    ys, xs = np.nonzero(bad)
    y, x = ys[0], xs[0]
    return ("%d pixels differ; first (%d,%d): img err %.3g T err %.3g last gpu %d oracle %d" %
            (bad.sum(), x, y, img_err[y, x], T_err[y, x], gpu["last"][y, x], ofw["last"][y, x]))


def check_backward(scene, gpu, obw, splat_mask=None):
    n = scene.n
    sel = np.ones(n, bool) if splat_mask is None else splat_mask
    g = obw["grads"]
    sl = obw["slack"]
    report = {}
    fields = GRAD_FIELDS + ((DIST_FIELD,) if gpu.get(DIST_FIELD) is not None else ())
    for k in fields:
        ref = g[k].reshape(n, -1)
        got = gpu[k].reshape(n, -1).astype(np.float64)
        slack = sl[k].reshape(n, -1) if sl is not None else 0.0
        tol = max(1e-4, 1e-3 * np.abs(ref[sel]).max(initial=0.0)) + slack
        err = np.abs(got - ref)
        bad = (err > tol) & sel[:, None]
        assert not bad.any(), "%s: %d elements off; worst err %.3g tol %.3g (ref %.3g got %.3g)" % (
            k, bad.sum(), err[bad].max(), np.broadcast_to(tol, err.shape)[bad][np.argmax(err[bad])],
            ref[bad][np.argmax(err[bad])], got[bad][np.argmax(err[bad])])
        report[k] = float((err[sel] / np.maximum(np.broadcast_to(tol, err.shape)[sel], 1e-30)).max(
            initial=0.0))
    if gpu["accum"] is not None:
        ref = g["accum"]
        tol = np.maximum(1e-5, obw["accum_err"]) + 2.0 ** -23 * np.abs(ref)
        if sl is not None:
            tol = tol + sl["accum"]
        err = np.abs(gpu["accum"].astype(np.float64) - ref)
        bad = (err > tol) & sel
        assert not bad.any(), "accum: %d off; worst %.3g" % (bad.sum(), err[bad].max())
        report["accum"] = float((err[sel] / tol[sel]).max(initial=0.0))
    return report


def _dist_grad(scene):
    return scene.dL_ddist if getattr(scene, "distortion", False) else None


def full_parity(scene, capacity=None, knife_cap=None, graph=False, threads=None, path=None):
    """Every output of the whole path against the oracle, every pixel and
    every splat.  The oracle runs tile-parallel on the host's cores
    (oracle.forward / oracle.backward with threads > 1: the same per-pixel
    code on disjoint tile sets).  graph=True runs the step the way bench.py
    times it (run_gpu_graph); path="splats" through the entry points that
    take the splats themselves (run_gpu_splats), path="nomask" with the
    backward given no blend masks (run_gpu_nomask)."""
    threads = oracle.default_threads() if threads is None else threads
    if path == "splats":
        gpu = run_gpu_splats(scene)
    elif path == "nomask":
        gpu = run_gpu_nomask(scene)
    else:
        gpu = run_gpu_graph(scene) if graph else run_gpu(scene, capacity)
    tl = check_pairs(scene, gpu)
    ofw = oracle.forward(scene, tl["vals"], tl["offs"], alt_capacity=1 << 20, threads=threads)
    f = check_forward(scene, gpu, ofw, knife_cap=knife_cap)
    s = check_weight_stats(scene, gpu, ofw)
    obw = oracle.backward(scene, tl["vals"], tl["offs"], dL_ddist=_dist_grad(scene),
                          threads=threads)
    b = check_backward(scene, gpu, obw)
    return {"fwd": f, "stats": s, "bwd": b, "pairs": tl["count"]}
