"""Parity of the CUDA path against the CPU oracle on the GPU (through the C ABI).

Every workload is compared in full -- every pair, the sorted order, the
offsets, every pixel of the forward and every splat's gradients -- the
2M-splat ones (4-6) at their full size, workloads 4 and 6 also in the launch
configuration bench.py times (the captured CUDA graph); the oracle runs
tile-parallel on the host's cores.  Knife-edge pixels (a float32 decision
within the oracle's error bound of its threshold) stay below 1e-4 of the
pixels on workloads 1-3; on the 2M-splat workloads, whose pixels blend ~70
splats each, the sound bound on the float32 transmittance grows with the
chain and they stay below 5e-4.  Edge cases cover empty and culled inputs,
ragged and tiny images, huge and off-screen splats, equal depths, dense
tiles, the alpha cap, a background, every combination of the four flags and
the pair-capacity overflow path.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import parity
    return parity


@pytest.mark.parametrize("wl", [1, 2, 3])
def test_workload_full_parity(P, wl):
    r = P.full_parity(synth.make_scene(wl), knife_cap=P.KNIFE_EDGE_CAP)
    print("workload", wl, r)


@pytest.mark.parametrize("wl,graph", [(4, False), (4, True), (5, False), (6, True)],
                         ids=["4-sync", "4-graph", "5-sync", "6-graph"])
def test_workload_full_size_full_parity(P, wl, graph):
    """The 2M-splat workloads compared in full: every pixel, every splat.
    graph=True: through the captured CUDA graph with the pair count on the
    device and 2.5 n pair buffers -- the launches bench.py times."""
    r = P.full_parity(synth.make_scene(wl), knife_cap=P.KNIFE_EDGE_CAP_DENSE, graph=graph)
    print("workload", wl, "graph" if graph else "sync", r)


@pytest.mark.parametrize("wl", [1, 2, 3, 4])
def test_entry_points_that_take_the_splats(P, wl):
    """ss_raster_fwd / ss_raster_bwd, given the splats themselves (the
    forward computes each batch's records; the backward rebuilds the records
    and re-evaluates the forward's blend decisions in its workspace, then
    replays transmittance), against the oracle in full."""
    sc = synth.make_scene(wl)
    sc.weight_stats = sc.distortion = False
    cap = P.KNIFE_EDGE_CAP if wl < 4 else P.KNIFE_EDGE_CAP_DENSE
    r = P.full_parity(sc, knife_cap=cap, path="splats")
    print("workload", wl, "from the splats", r)


@pytest.mark.parametrize("accum,median", [(False, False), (True, True), (False, True)])
def test_entry_points_that_take_the_splats_flags(P, accum, median):
    sc = _scene(96, 80, 500, seed=19, wl=2)
    sc.accum_weight, sc.median_depth = accum, median
    P.full_parity(sc, path="splats")


@pytest.mark.parametrize("wl", [2, 3, 5, 6])
def test_backward_without_the_forwards_blend_masks(P, wl):
    """ss_raster_bwd_records given no blend masks re-evaluates the decisions
    (every variant: workload 5 has the median and the weight statistics,
    workload 6 the distortion), against the oracle in full."""
    cap = P.KNIFE_EDGE_CAP if wl < 4 else P.KNIFE_EDGE_CAP_DENSE
    r = P.full_parity(synth.make_scene(wl), knife_cap=cap, path="nomask")
    print("workload", wl, "no masks", r)


@pytest.mark.parametrize("W,H", [(37, 23), (1, 1), (17, 1), (129, 65)])
def test_entry_points_that_take_the_splats_on_ragged_images(P, W, H):
    sc = _scene(W, H, 80, seed=W * 1000 + H + 7)
    sc.weight_stats = sc.distortion = False
    sc.mean2d[:, 0] = sc.mean2d[:, 0] * 1.2 - 0.1 * W
    sc.mean2d[:, 1] = sc.mean2d[:, 1] * 1.2 - 0.1 * H
    P.full_parity(sc, path="splats")
    P.full_parity(sc, path="nomask")


def test_workload_3_with_distortion(P):
    sc = synth.make_scene(3)
    sc.distortion = True
    r = P.full_parity(sc)
    print("workload 3 + distortion", r)


def _scene(W, H, n, seed=0, wl=1, **over):
    sc = synth.make_scene(wl, seed=seed, n=n, W=W, H=H)
    for k, v in over.items():
        setattr(sc, k, v)
    return sc


@pytest.mark.parametrize("W,H", [(37, 23), (1, 1), (16, 16), (17, 1), (1, 300), (129, 65)])
def test_ragged_and_tiny_images(P, W, H):
    sc = _scene(W, H, 80, seed=W * 1000 + H)
    sc.mean2d[:, 0] = sc.mean2d[:, 0] * 1.2 - 0.1 * W
    sc.mean2d[:, 1] = sc.mean2d[:, 1] * 1.2 - 0.1 * H
    P.full_parity(sc)


def test_no_splats(P):
    sc = _scene(40, 30, 0)
    gpu = P.run_gpu(sc)
    assert gpu["count"] == 0
    assert np.all(gpu["offs"] == 0)
    assert np.all(gpu["T_final"] == 1.0) and np.all(gpu["last"] == 0)
    assert np.all(gpu["image"] == 0.0)


def test_all_culled(P):
    sc = _scene(48, 48, 100, seed=3)
    sc.depth[:] = -1.0
    gpu = P.run_gpu(sc)
    assert gpu["count"] == 0 and gpu["culled"] == 100
    assert all(np.all(gpu[k] == 0) for k in P.GRAD_FIELDS)


def test_invalid_inputs_are_culled(P):
    sc = _scene(64, 64, 200, seed=4)
    sc.depth[::7] = 0.0
    sc.conic[1::11, 1] = 5.0           # indefinite
    sc.opacity[2::13] = 1e-3           # below 1/255
    sc.mean2d[3::17, 0] = np.inf
    sc.rgb[5::19, 2] = np.nan
    P.full_parity(sc)


def test_huge_and_offscreen_splats(P):
    sc = _scene(100, 70, 60, seed=5)
    sc.conic[:10] = synth.conic_from_scales(np.zeros(10), np.full(10, 40.0),
                                            np.full(10, 25.0)).astype(np.float32)
    sc.mean2d[10:20] += np.float32([500.0, 0.0])
    sc.mean2d[20:30] -= np.float32([0.0, 300.0])
    sc.mean2d[30:35] = np.float32([-20.0, -20.0])
    P.full_parity(sc)


def test_equal_depths_tie_break_by_index(P):
    sc = _scene(64, 64, 400, seed=6)
    sc.depth[:] = np.float32(3.0)
    sc.depth[::3] = np.float32(2.0)
    P.full_parity(sc)


def test_dense_single_tile_many_batches(P):
    """3000 splats in one tile: many 256-splat batches, early termination."""
    sc = _scene(16, 16, 3000, seed=7)
    sc.opacity[:] = np.float32(0.05)
    P.full_parity(sc)
    sc.opacity[:] = np.float32(0.02)   # survives deep into the list
    P.full_parity(sc)


def test_alpha_cap_and_background(P):
    sc = _scene(64, 48, 150, seed=8)
    sc.opacity[:40] = np.float32(1.0)   # alpha capped at 0.99 near their centres
    sc.bg = np.float32([0.25, 0.5, 0.75])
    P.full_parity(sc)


@pytest.mark.parametrize("flags", range(16))
def test_flag_variants(P, flags):
    """Every combination of accumulated weight, median depth, weight
    statistics and distortion."""
    accum, median, stats, dist = [bool(flags >> k & 1) for k in range(4)]
    sc = _scene(96, 80, 500, seed=9, wl=2)
    sc.accum_weight, sc.median_depth, sc.weight_stats, sc.distortion = accum, median, stats, dist
    r = P.full_parity(sc)
    assert (r["stats"] is not None) == stats
    assert ("ddepth" in r["bwd"]) == dist
    if stats:
        assert r["stats"]["blended"] > 100


def test_distortion_dense_tile_and_far_depths(P):
    """3,000 splats on one tile with depths over [1, 100]: long per-pixel
    lists and totals whose terms are far larger than the distortion."""
    sc = _scene(16, 16, 3000, seed=12)
    sc.opacity[:] = np.float32(0.02)
    sc.depth[:] = np.float32(1.0) + np.float32(99.0) * np.random.default_rng(3).random(
        sc.n).astype(np.float32)
    sc.distortion = True
    sc.dL_ddist = np.random.default_rng(4).normal(0, 1e-5, (sc.H, sc.W)).astype(np.float32)
    P.full_parity(sc)


def test_weight_stats_with_dense_overlap(P):
    """Many splats over one tile: the per-warp reductions see up to 32
    blending lanes and the atomics many warps per splat."""
    sc = _scene(16, 16, 3000, seed=7)
    sc.opacity[:] = np.float32(0.02)
    sc.weight_stats = True
    r = P.full_parity(sc)
    assert r["stats"]["blended"] > 1000


def test_capacity_overflow_reports_and_recovers(P):
    import torch
    import gaussian_splatting_differentiable_gb300 as ss
    sc = _scene(128, 128, 400, seed=10, wl=2)
    sp = ss.Splats.from_numpy(sc)
    keys = torch.full((50,), -1, dtype=torch.int64, device="cuda")
    vals = torch.full((50,), -1, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(ss.COUNTER_WORDS, dtype=torch.int64, device="cuda")
    recs = torch.empty(ss.ss_record_bytes(sc.n), dtype=torch.uint8, device="cuda")
    ss.ss_bin_tiles(sp, sc.W, sc.H, keys, vals, 40, cnt, recs)
    st, pairs, culled = ss.ss_pair_count(cnt, 40)
    import oracle
    assert st == ss.SS_ERR_CAPACITY and pairs == oracle.tile_lists(sc)["count"] > 40
    # nothing written past the capacity
    assert torch.all(keys[40:] == -1) and torch.all(vals[40:] == -1)
    assert "capacity" in ss.ss_last_error()
    P.full_parity(sc, capacity=pairs)


def test_two_calls_in_a_row_agree(P):
    sc = synth.make_scene(2)
    a = P.run_gpu(sc)
    b = P.run_gpu(sc)
    for k in ("keys", "vals", "offs", "image", "T_final", "last", "accum"):
        assert np.array_equal(a[k], b[k]), k


def test_profile_counts_every_launch(P):
    import torch
    import gaussian_splatting_differentiable_gb300 as ss
    sc = synth.make_scene(2)
    sp = ss.Splats.from_numpy(sc)
    r = ss.Rasterizer(sc.W, sc.H, sc.n, 4 * sc.n, ss.SS_ACCUM_WEIGHT, device="cuda")
    dL = torch.from_numpy(sc.dL_dimage).cuda()
    ss.ss_profile_collect()
    ss.ss_profile_enable(True)
    r.step(sp, dL)
    r.step(sp, dL)
    ss.ss_profile_enable(False)
    prof = ss.ss_profile_collect()
    assert prof["k_emit_pairs"][0] == 2 and prof["k_raster_bwd"][0] == 2
    assert prof["k_sort_pass"][0] == 2 * 5   # 8 tile bits + 32 depth bits -> 5 digits
    assert prof["k_sort_final"][0] == 2 and prof["k_sort_ties"][0] == 2
    assert all(v[1] > 0 for v in prof.values())
    assert ss.ss_profile_collect() == {}


def _snapshot(r):
    import torch
    torch.cuda.synchronize()
    return {"offs": r.tile_offsets.cpu().numpy().copy(), "image": r.image.cpu().numpy().copy(),
            "T": r.T_final.cpu().numpy().copy(), "last": r.last_contrib.cpu().numpy().copy(),
            **{k: v.cpu().numpy().copy() for k, v in r.grads.items()},
            "accum": r.accum_weight.cpu().numpy().copy()}


def _same(a, b, P):
    for k in ("offs", "image", "T", "last", "accum"):
        assert np.array_equal(a[k], b[k]), k
    for k in P.GRAD_FIELDS:
        tol = max(1e-4, 1e-3 * np.abs(a[k]).max())
        assert np.abs(a[k] - b[k]).max() <= tol, k


def test_device_count_step_and_graph_replay_match_synced_step(P):
    """bin -> sort on the device count -> fwd -> bwd without a host read, and a
    CUDA graph of it, give what the synchronised path gives."""
    import torch
    import gaussian_splatting_differentiable_gb300 as ss
    sc = synth.make_scene(3)
    sp = ss.Splats.from_numpy(sc)
    dL = torch.from_numpy(sc.dL_dimage).cuda()
    r = ss.Rasterizer(sc.W, sc.H, sc.n, 16, ss.SS_ACCUM_WEIGHT)
    r.step(sp, dL)                      # grows the pair buffers
    ref = _snapshot(r)
    r.step_async(sp, dL)
    r.check()
    _same(ref, _snapshot(r), P)
    g = r.capture(sp, dL)
    for _ in range(2):
        r.image.zero_()
        g.replay()
        r.check()
        _same(ref, _snapshot(r), P)


def test_device_count_sort_reports_capacity_overflow(P):
    import torch
    import gaussian_splatting_differentiable_gb300 as ss
    sc = synth.make_scene(2)
    sp = ss.Splats.from_numpy(sc)
    r = ss.Rasterizer(sc.W, sc.H, sc.n, 1000, 0)    # far fewer than the ~18k pairs
    ss.ss_bin_tiles(sp, sc.W, sc.H, r.keys, r.vals, r.capacity, r.counters, r.records)
    ss.ss_sort_pairs_dev(r.keys, r.vals, r.counters, r.capacity, sc.W, sc.H, r.tile_offsets,
                         r.workspace)
    assert ss.ss_sort_status(r.workspace) == ss.SS_ERR_CAPACITY
    offs = r.tile_offsets.cpu().numpy().view(np.uint32)
    assert offs[-1] == 1000 and np.all(np.diff(offs.astype(np.int64)) >= 0)


def test_device_count_sort_of_no_pairs(P):
    import torch
    import gaussian_splatting_differentiable_gb300 as ss
    sc = _scene(40, 30, 50, seed=12)
    sc.depth[:] = -1.0                 # every splat culled: zero pairs
    sp = ss.Splats.from_numpy(sc)
    r = ss.Rasterizer(sc.W, sc.H, sc.n, 64, 0)
    r.tile_offsets.fill_(7)
    ss.ss_bin_tiles(sp, sc.W, sc.H, r.keys, r.vals, r.capacity, r.counters, r.records)
    ss.ss_sort_pairs_dev(r.keys, r.vals, r.counters, r.capacity, sc.W, sc.H, r.tile_offsets,
                         r.workspace)
    assert ss.ss_sort_status(r.workspace) == ss.SS_OK
    assert np.all(r.tile_offsets.cpu().numpy() == 0)


def _bin_for_sort(sc, cap_factor=8):
    import gaussian_splatting_differentiable_gb300 as ss
    sp = ss.Splats.from_numpy(sc)
    r = ss.Rasterizer(sc.W, sc.H, sc.n, cap_factor * sc.n, 0)
    ss.ss_bin_tiles(sp, sc.W, sc.H, r.keys, r.vals, r.capacity, r.counters, r.records)
    st, n, _ = ss.ss_pair_count(r.counters, r.capacity)
    assert st == ss.SS_OK
    keys = r.keys[:n].cpu().numpy().view(np.uint64).copy()
    vals = r.vals[:n].cpu().numpy().view(np.uint32).copy()
    return r, n, keys, vals


@pytest.mark.parametrize("kind", ["wide", "narrow", "equal", "three_values", "narrow_1024_tiles"])
def test_device_count_sort_over_the_recorded_depth_range(P, kind):
    """The device-count sort takes its digits from (tile, depth bits - lo)
    on the bits the recorded depth range needs (fewer passes when the range
    is narrow); the order must still be (key, value): checked against a
    lexsort of the binned pairs, with the range the binning recorded
    checked against the splats that have pairs."""
    import gaussian_splatting_differentiable_gb300 as ss
    # 300 x 200 has 247 tiles (8 tile bits: 3 passes for a narrow range, 5
    # for the wide one); 512 x 512 has 1,024 (10 bits: 4 passes, an even
    # count, for a narrow range)
    sc = _scene(512, 512, 20000, seed=21) if kind == "narrow_1024_tiles" else \
        _scene(300, 200, 20000, seed=21)
    rng = np.random.default_rng(21)
    if kind == "wide":        # every exponent from 1e-3 to 1e5: all 32 depth bits
        sc.depth[:] = (10.0 ** rng.uniform(-3, 5, sc.n)).astype(np.float32)
    elif kind in ("narrow", "narrow_1024_tiles"):    # a few ulps apart: the 16-bit minimum
        sc.depth[:] = rng.uniform(2.0, 2.001, sc.n).astype(np.float32)
    elif kind == "equal":
        sc.depth[:] = np.float32(3.0)
    else:
        sc.depth[:] = rng.choice(np.float32([1.5, 7.25, 40.0]), sc.n)
    r, n, keys, vals = _bin_for_sort(sc)
    cnt = r.counters.cpu().numpy().view(np.uint64)
    dbits = sc.depth.view(np.uint32)[vals]
    assert cnt[2] == dbits.min() and cnt[3] == dbits.max()
    ss.ss_sort_pairs_dev(r.keys, r.vals, r.counters, r.capacity, sc.W, sc.H, r.tile_offsets,
                         r.workspace)
    assert ss.ss_sort_status(r.workspace) == ss.SS_OK
    order = np.lexsort((vals, keys))
    assert np.array_equal(r.keys[:n].cpu().numpy().view(np.uint64), keys[order])
    assert np.array_equal(r.vals[:n].cpu().numpy().view(np.uint32), vals[order])
    tiles = ((sc.W + 15) // 16) * ((sc.H + 15) // 16)
    want = np.searchsorted(keys[order] >> np.uint64(32), np.arange(tiles + 1, dtype=np.uint64))
    assert np.array_equal(r.tile_offsets.cpu().numpy().view(np.uint32), want.astype(np.uint32))


def test_device_count_sort_flags_a_depth_outside_the_recorded_range(P):
    """Counters whose range leaves out some pair's depth (not the binning's
    own) make the sort report SS_ERR_DEVICE instead of a wrong order."""
    import gaussian_splatting_differentiable_gb300 as ss
    sc = _scene(64, 64, 2000, seed=22)
    sc.depth[:] = np.linspace(1.0, 100.0, sc.n, dtype=np.float32)
    r, n, keys, vals = _bin_for_sort(sc)
    hi = int(r.counters[3].item())
    r.counters[2] = (hi - (1 << 20)) & ~0xffff      # above the smallest depths' bits
    ss.ss_sort_pairs_dev(r.keys, r.vals, r.counters, r.capacity, sc.W, sc.H, r.tile_offsets,
                         r.workspace)
    assert ss.ss_sort_status(r.workspace) == ss.SS_ERR_DEVICE


def test_long_runs_of_equal_depths_sort_bit_exact(P):
    """40,000 small splats on 2x2 tiles, a quarter of them at one depth: runs
    of ~2,500 equal keys per tile, ordered by splat index by the long-run
    radix sort (a quadratic insertion sort would take seconds), compared
    pair by pair."""
    import synth
    sc = _scene(32, 32, 40000, seed=13)
    sc.depth[::4] = np.float32(5.0)
    gpu = P.run_gpu(sc, capacity=8 * sc.n)
    tl = P.check_pairs(sc, gpu)
    assert np.diff(tl["offs"]).max() > 8192


@pytest.mark.parametrize("case", ["packed_odd_passes", "packed_even_passes", "unpacked",
                                  "packed_long_runs"])
def test_sort_modes_against_the_oracle(P, case):
    """The passes move one 64-bit word (key bits << value bits | value) when
    the sorted key bits and the largest value fit in 64 bits together, else a
    key and a value; the packed words ping-pong so that the last pass lands
    in the alternate buffer, through a third buffer when the pass count is
    even.  Synthetic pairs reach each mode: 256 tiles (40 key bits, 5
    passes), 1,024 tiles (42 bits, 6 passes), 31-bit values (73 bits: not
    packed), and runs of 3,000 equal keys (the long-run sort after
    unpacking).  Compared with the oracle's sort and offsets."""
    import torch
    import oracle
    import gaussian_splatting_differentiable_gb300 as ss
    W, H = (256, 256) if case == "packed_odd_passes" else (512, 512)
    tiles = ((W + 15) // 16) * ((H + 15) // 16)
    n = 50000
    rng = np.random.default_rng(["packed_odd_passes", "packed_even_passes", "unpacked",
                                 "packed_long_runs"].index(case) + 31)
    tile = rng.integers(0, tiles, n).astype(np.uint64)
    dbits = rng.integers(0x3F800000, 0x42C80000, n).astype(np.uint64)
    vmax = (1 << 31) - 1 if case == "unpacked" else (1 << 20) - 1
    vals = rng.integers(0, vmax + 1, n).astype(np.uint32)
    vals[0] = vmax
    if case == "packed_long_runs":
        tile[: 2 * 3000] = 7
        dbits[:3000] = 0x40400000
        dbits[3000: 2 * 3000] = 0x40A00000
    keys = (tile << np.uint64(32)) | dbits
    k_d = torch.from_numpy(keys.view(np.int64)).cuda()
    v_d = torch.from_numpy(vals.view(np.int32)).cuda()
    offs = torch.zeros(tiles + 1, dtype=torch.int32, device="cuda")
    ws = torch.empty(ss.ss_workspace_bytes(0, n, W, H), dtype=torch.uint8, device="cuda")
    ss.ss_sort_pairs(k_d, v_d, n, W, H, offs, ws)
    assert ss.ss_sort_status(ws) == ss.SS_OK
    want_k, want_v = oracle.sort_pairs(keys, vals)
    assert np.array_equal(k_d.cpu().numpy().view(np.uint64), want_k)
    assert np.array_equal(v_d.cpu().numpy().view(np.uint32), want_v)
    assert np.array_equal(offs.cpu().numpy().view(np.uint32), oracle.offsets(want_k, tiles))


def test_forward_clears_the_backward_records(P):
    """ss_raster_fwd_records with bwd_workspace clears the backward's gradient
    records and ss_raster_bwd_records with SS_RECORDS_CLEARED skips its own
    clearing pass:
    the result equals that of a backward that clears them itself (gradients
    to float-atomic ordering, the fixed-point weight bit for bit), although
    the workspace started as non-zero bytes and the sort wrote over the
    records' bytes.  A flagged backward on records that nobody cleared adds
    to the old sums (the weight doubles), so the check is not vacuous."""
    import torch
    import gaussian_splatting_differentiable_gb300 as ss
    sc = synth.make_scene(2)
    sp = ss.Splats.from_numpy(sc)
    r = ss.Rasterizer(sc.W, sc.H, sc.n, 4 * sc.n, ss.SS_ACCUM_WEIGHT, device="cuda")
    dL = torch.from_numpy(sc.dL_dimage).cuda()
    r.workspace.fill_(0x7f)
    r.bin_and_sort(sp)
    r.forward(sp)
    r.backward(sp, dL)            # flagged: the forward cleared the records
    a = {k: v.clone() for k, v in r.grads.items()}
    wa = r.accum_weight.clone()
    args = (r.records, r.n, r.vals, r.tile_offsets, r.n_pairs, sc.W, sc.H, r.bg)
    rest = (r.T_final, r.last_contrib, r.blend_masks, dL, r.grads, r.accum_weight, r.workspace)
    ss.ss_raster_bwd_records(*args, r.flags, *rest)      # clears them itself
    torch.cuda.synchronize()
    assert torch.equal(r.accum_weight, wa)
    for k, v in a.items():
        tol = max(1e-4, 1e-3 * float(v.abs().max()))
        assert float((r.grads[k] - v).abs().max()) <= tol, k
    ss.ss_raster_bwd_records(*args, r.flags | ss.SS_RECORDS_CLEARED, *rest)   # stale sums kept
    torch.cuda.synchronize()
    assert torch.equal(r.accum_weight, 2 * wa)


def test_step_pipeline_matches_single_steps(P):
    """ss.StepPipeline (double-buffered copies in and out around the step's
    graph) returns what a synchronous step computes: the image and the
    accumulated weight bit for bit, gradients to float-atomic reordering."""
    import torch
    import gaussian_splatting_differentiable_gb300 as ss
    sc = synth.make_scene(2)
    host_in = {k: torch.from_numpy(getattr(sc, k)).pin_memory() for k in ss.StepPipeline.KEYS}
    host_dL = torch.from_numpy(sc.dL_dimage).pin_memory()
    pipe = ss.StepPipeline(sc.W, sc.H, sc.n, ss.SS_ACCUM_WEIGHT, host_in, host_dL, device="cuda")
    outs = [pipe.host_output_buffers(), pipe.host_output_buffers()]
    pipe.run(5, host_in, host_dL, outs)
    pipe.check()
    r = ss.Rasterizer(sc.W, sc.H, sc.n, 4 * sc.n, ss.SS_ACCUM_WEIGHT, device="cuda")
    r.step(ss.Splats.from_numpy(sc), torch.from_numpy(sc.dL_dimage).cuda())
    torch.cuda.synchronize()
    ref = [r.image] + [r.grads[k] for k in ("dmean2d", "dconic", "dopacity", "drgb")] + \
        [r.accum_weight]
    for host in outs:
        got = [h.numpy() for h in host]
        refn = [t.cpu().numpy() for t in ref]
        assert np.array_equal(got[0], refn[0])              # image
        assert np.array_equal(got[-1], refn[-1])            # accumulated weight (fixed point)
        for g, e in zip(got[1:-1], refn[1:-1]):
            assert np.abs(g - e).max() <= 1e-5 * max(np.abs(e).max(), 1e-30)


@pytest.mark.parametrize("seed", range(12))
def test_random_scenes(P, seed):
    """Seeded random configurations: image size, splat count, scale,
    opacity (up to the alpha cap) and depth ranges (with equal-depth
    clusters), background and every output flag drawn at random, each
    compared in full with the oracle."""
    rng = np.random.default_rng(1000 + seed)
    W, H = int(rng.integers(1, 200)), int(rng.integers(1, 200))
    n = int(rng.integers(0, 3000))
    lo = float(rng.uniform(0.2, 2.0))
    wl = synth.Workload("random", W, H, n, (lo, lo * float(rng.uniform(1.0, 8.0))),
                        (float(rng.uniform(0.004, 0.5)), float(rng.uniform(0.5, 1.0))),
                        (1.0, float(rng.uniform(1.5, 200.0))), float(rng.uniform(0.01, 1.0)),
                        bool(rng.integers(2)), bool(rng.integers(2)),
                        weight_stats=bool(rng.integers(2)), distortion=bool(rng.integers(2)))
    sc = synth.make_scene(wl, seed=seed)
    if n and rng.integers(2):
        k = max(1, n // 5)
        sc.depth[rng.choice(n, k, replace=False)] = np.float32(rng.uniform(1, 5))
    sc.bg = rng.uniform(0, 1, 3).astype(np.float32)
    r = P.full_parity(sc)
    print(seed, W, H, n, r["pairs"])


@pytest.mark.parametrize("W,H", [(32768, 40), (40, 32768)])
def test_maximum_side_length(P, W, H):
    """The longest image side the ABI accepts (32,768 px), with a ragged
    other side: 2,048 x 3 tiles (13 tile-id bits), compared in full."""
    sc = _scene(W, H, 4000, seed=14, wl=3)
    r = P.full_parity(sc)
    assert r["pairs"] > 4000


def test_both_forms_of_the_entry_points_agree(P):
    """ss_raster_fwd (records computed in the kernel from the splats) and
    ss_raster_fwd_records (the binning's records) give the same image, T and
    last contributor bit for bit -- the records are the same bits; the two
    backwards (rebuilt records and re-evaluated decisions against the
    forward's masks) the same accumulated weight bit for bit (fixed point)
    and the same gradients up to float-atomic ordering."""
    import torch
    import gaussian_splatting_differentiable_gb300 as ss
    sc = synth.make_scene(3)
    flags = ss.SS_ACCUM_WEIGHT
    sp = ss.Splats.from_numpy(sc)
    dL = torch.from_numpy(sc.dL_dimage).cuda()
    r = ss.Rasterizer(sc.W, sc.H, sc.n, 4 * sc.n, flags, bg=sc.bg)
    r.bin_and_sort(sp)
    r.forward(sp)
    r.backward(sp, dL)
    torch.cuda.synchronize()
    ref = {"image": r.image.clone(), "T": r.T_final.clone(), "last": r.last_contrib.clone(),
           "accum": r.accum_weight.clone(), **{k: v.clone() for k, v in r.grads.items()}}
    img, T, last = torch.empty_like(r.image), torch.empty_like(r.T_final), \
        torch.empty_like(r.last_contrib)
    ss.ss_raster_fwd(sp, r.vals, r.tile_offsets, sc.W, sc.H, r.bg, flags, img, T, last)
    grads = {k: torch.empty_like(v) for k, v in r.grads.items()}
    acc = torch.empty_like(r.accum_weight)
    ss.ss_raster_bwd(sp, r.vals, r.tile_offsets, sc.W, sc.H, r.bg, flags, T, last, dL, grads, acc,
                     r.workspace)
    torch.cuda.synchronize()
    assert ss.ss_sort_status(r.workspace) == ss.SS_OK
    assert torch.equal(img, ref["image"]) and torch.equal(T, ref["T"])
    assert torch.equal(last, ref["last"]) and torch.equal(acc, ref["accum"])
    for k, v in grads.items():
        tol = max(1e-4, 1e-3 * float(ref[k].abs().max()))
        assert float((v - ref[k]).abs().max()) <= tol, k


def test_backward_from_the_splats_reports_a_workspace_too_small_for_its_masks(P):
    """ss_raster_bwd learns the pair count only on the device: given a
    workspace whose mask rows hold fewer pairs than the lists, it writes and
    reads only inside the rows and reports SS_ERR_CAPACITY through the
    status word (the gradients are then not valid)."""
    import torch
    import gaussian_splatting_differentiable_gb300 as ss
    sc = synth.make_scene(2)
    flags = ss.SS_ACCUM_WEIGHT
    sp = ss.Splats.from_numpy(sc)
    dL = torch.from_numpy(sc.dL_dimage).cuda()
    r = ss.Rasterizer(sc.W, sc.H, sc.n, 4 * sc.n, flags, bg=sc.bg)
    pairs = r.bin_and_sort(sp)
    ss.ss_raster_fwd(sp, r.vals, r.tile_offsets, sc.W, sc.H, r.bg, flags, r.image, r.T_final,
                     r.last_contrib)
    small = ss.ss_workspace_bytes(sc.n, pairs // 2, sc.W, sc.H)
    ws = torch.empty(small, dtype=torch.uint8, device="cuda")
    ws[:4].zero_()   # a clean status word (no sort ran on this buffer)
    ss.ss_raster_bwd(sp, r.vals, r.tile_offsets, sc.W, sc.H, r.bg, flags, r.T_final,
                     r.last_contrib, dL, r.grads, r.accum_weight, ws)
    assert ss.ss_sort_status(ws) == ss.SS_ERR_CAPACITY
    ws2 = torch.empty(ss.ss_workspace_bytes(sc.n, pairs, sc.W, sc.H), dtype=torch.uint8,
                      device="cuda")
    ws2[:4].zero_()
    ss.ss_raster_bwd(sp, r.vals, r.tile_offsets, sc.W, sc.H, r.bg, flags, r.T_final,
                     r.last_contrib, dL, r.grads, r.accum_weight, ws2)
    assert ss.ss_sort_status(ws2) == ss.SS_OK
