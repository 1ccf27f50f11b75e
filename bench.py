#!/usr/bin/env python
"""Benchmark of the splat rasterization path on the 2M-splat, 1237x822 workload.

One step = the whole path over one scene: tile binning, onesweep sort +
tile ranges on the device-side pair count, forward, backward, replayed as
one CUDA graph (per-kernel times come from a second timed pass of the same
step launched without the graph).  Prints one JSON
line (rank 0).  Under torchrun each rank runs an independent replica (the path
does not shard across GPUs here); value = all ranks' candidate splat-pixel
pairs / the slowest rank's time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (test infrastructure) on the host
cores, on a bounded sample of the same workload, in the same metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "rasterize_bwd ms/call and splat-pixel pairs/s at 2M splats 1237×822; % roofline"
UNIT = "splat-px pairs/s"
WORKLOAD = 4
L2_FLUSH_BYTES = 256 << 20
# The backward kernel's source, as the committed ncu counters are tied to it:
# ss_bwd.cu up to the end of k_raster_bwd (the line defining kBwdDynSmem; the
# launch code and the other kernels of the file follow it), and the headers
# it compiles with.
BWD_SOURCES = (("gaussian_splatting_differentiable_gb300/csrc/ss_bwd.cu", "constexpr int kBwdDynSmem"),
               ("gaussian_splatting_differentiable_gb300/csrc/ss_device.cuh", None),
               ("gaussian_splatting_differentiable_gb300/csrc/ss_internal.h", None))


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-next", action="store_true", help="skip the projection / SSIM legs")
    ap.add_argument("--only", choices=["projection", "ssim", "distortion"],
                    help="run one leg of the next rows alone and print its JSON (for profiling)")
    return ap.parse_args()


def candidate_pairs(offs: np.ndarray, W: int, H: int) -> int:
    """sum over tiles of (pairs of the tile) x (pixels of the tile inside the image)."""
    tx, ty = (W + 15) // 16, (H + 15) // 16
    per = np.diff(offs.astype(np.int64)).reshape(ty, tx)
    wx = np.minimum(16, W - 16 * np.arange(tx))
    wy = np.minimum(16, H - 16 * np.arange(ty))
    return int((per * wy[:, None] * wx[None, :]).sum())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [r for (t, r) in self.rows if self.t0 is not None and self.t0 - 0.06 <= t <= (self.t1 or t) + 0.06]
        if not rows:
            rows = [r for (_, r) in self.rows]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[2]))
                mx.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for nm, v in zip(names, r[6:10]):
                if v.strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle

def cpu_description() -> dict:
    """The host's logical CPUs and CPU (x86: the model name; Arm: the
    implementer and part numbers /proc/cpuinfo lists)."""
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                k, v = k.strip(), v.strip()
                if k in ("model name", "CPU implementer", "CPU part") and v and k not in fields:
                    fields[k] = v
    except OSError:
        pass
    import platform
    if "model name" in fields:
        model = fields["model name"]
    elif "CPU part" in fields:
        model = "%s, CPU implementer %s, CPU part %s" % (
            platform.machine(), fields.get("CPU implementer", "?"), fields["CPU part"])
    else:
        model = platform.processor() or platform.machine()
    return {"nproc": os.cpu_count(), "model": model}


def oracle_bin_sort(scene):
    """The oracle's binning, sort and tile ranges of the whole scene
    (single-threaded C)."""
    import oracle
    keys, vals, count, _ = oracle.bin_tiles(scene)
    keys, vals = oracle.sort_pairs(keys, vals)
    tx, ty = oracle.tiles_xy(scene.W, scene.H)
    return vals, oracle.offsets(keys, tx * ty)


def oracle_raster(scene, vals, offs, mask, threads: int, sums=None):
    """The oracle's forward and backward over the tiles of `mask`, split over
    `threads` host threads (tile-parallel; the per-pixel code as it stands).
    sums: per-thread gradient accumulators shared by successive calls."""
    import oracle
    oracle.forward(scene, vals, offs, tile_mask=mask, threads=threads)
    oracle.backward(scene, vals, offs, tile_mask=mask, slack=False, threads=threads, into=sums)


def oracle_pieces(scene, pieces: int, threads: int, warmup: int = 0):
    """One whole step of the oracle (bin + sort + forward + backward of every
    tile) timed in `pieces` consecutive pieces: piece 0 bins and sorts the
    scene and each piece composites and back-propagates its share of the
    tiles (oracle.tile_parts: equal work).  Nothing is extrapolated: the
    pieces together are the whole step.  Returns (piece seconds, details)."""
    import oracle
    vals, offs = oracle_bin_sort(scene)
    masks = oracle.tile_parts(scene.W, scene.H, offs, None, pieces)
    for k in range(warmup):
        oracle_raster(scene, vals, offs, masks[k % len(masks)], threads)
    sums = oracle.backward_sums(scene.n, threads, slack=False)   # zeroed before the timing
    times = []
    for k, m in enumerate(masks):
        t0 = time.perf_counter()
        if k == 0:
            vals, offs = oracle_bin_sort(scene)
        oracle_raster(scene, vals, offs, m, threads, sums)
        if k == len(masks) - 1:
            oracle.add_backward_sums(sums)        # the step's gradients
        times.append(time.perf_counter() - t0)
    return times, {"pieces": len(masks), "candidates": candidate_pairs(offs, scene.W, scene.H)}


def oracle_single_core_rate(scene, n_tiles: int, seed: int = 0) -> dict:
    """The single-threaded oracle's forward + backward rate on n_tiles random
    tiles (candidate pairs per second of rasterization; bin + sort excluded)."""
    import oracle
    vals, offs = oracle_bin_sort(scene)
    tx, ty = oracle.tiles_xy(scene.W, scene.H)
    rng = np.random.default_rng(seed)
    mask = np.zeros(tx * ty, np.uint8)
    mask[rng.choice(tx * ty, min(n_tiles, tx * ty), replace=False)] = 1
    t0 = time.perf_counter()
    oracle_raster(scene, vals, offs, mask, 1)
    dt = time.perf_counter() - t0
    per = np.diff(offs.astype(np.int64))
    wx = np.minimum(16, scene.W - 16 * (np.arange(tx * ty) % tx))
    wy = np.minimum(16, scene.H - 16 * (np.arange(tx * ty) // tx))
    cand = int((per * wx * wy)[mask.astype(bool)].sum())
    return {"value": cand / dt, "unit": UNIT, "cores": 1, "tiles": int(mask.sum()),
            "candidates": cand, "seconds": dt,
            "what": "forward + backward of %d random tiles, single-threaded" % int(mask.sum())}


def run_reference(args, rank: int):
    import oracle
    import synth
    if rank != 0:
        return
    scene = synth.make_scene(args.workload)
    threads = oracle.default_threads()
    times, det = oracle_pieces(scene, max(1, args.steps), threads, warmup=args.warmup)
    total = sum(times)
    steps = len(times)
    value = det["candidates"] / total
    sample = ("the %d timed steps are one whole step of the %d-splat scene: step 0 bins and "
              "sorts the scene (single-threaded) and each step runs the forward and backward "
              "of a 1/%d share of the tiles (equal work), tile-parallel on %d threads; %d "
              "warm-up steps ran a share each first" % (steps, scene.n, steps, threads,
                                                       args.warmup))
    cpu = cpu_description()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": synth.WORKLOADS[args.workload].name, "W": scene.W, "H": scene.H,
                       "splats": scene.n, "candidate_splat_px": det["candidates"]},
            "whole_step_ms": 1e3 * total,
            "host": cpu,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

def max_over_ranks(x: float, dist, device) -> float:
    """The largest x over all ranks (the slowest replica's time); x itself
    when not distributed."""
    if not dist:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, units_per_rank: float, ms: float) -> float:
    """Whole-job throughput: the units every replica processed over the
    slowest replica's time (replicas of the same step, weak scaling)."""
    return world * units_per_rank / (ms * 1e-3)


def source_sha(sources) -> str:
    """Hash of (path, end) pairs: each file up to and including the line
    that holds `end` (the whole file when end is None)."""
    h = hashlib.sha256()
    for p, end in sources:
        with open(os.path.join(ROOT, p), "rb") as f:
            data = f.read()
        if end is not None:
            i = data.index(end.encode())
            data = data[:data.index(b"\n", i) + 1]
        h.update(data)
    return h.hexdigest()[:16]


def recorded_counters(kernel: str, workload: str):
    """The committed ncu record of the kernel (profiles/traffic.json), if it
    was taken on the current source of the kernel and on this workload."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        rec = json.load(open(p)).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_sha") != source_sha(BWD_SOURCES):
        return None
    if rec.get("workload_name") != workload:
        return None
    return rec


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu record (None if stale)."""
    rec = recorded_counters(kernel, workload)
    return rec.get("dram_bytes_per_launch_full") if rec else None


# The backward's method minimum per blended (pixel, splat) pair, in thread
# instructions: the replay (the exponent from the splat's record: 2 sub,
# 2 mul, 2 fma; the exponential, o G and the cap: 3; T in front, 1 - alpha,
# its reciprocal and the product: 3; w = alpha T: 1; dL/dimage . rgb: 3;
# dL/dalpha: 2; q = dL/dsigma with the cap's select: 2; the suffix colour
# sum: 1 -- 21) and the pixel's share of the per-splat sums (q times 1, u,
# v, u^2, uv, v^2 and w times 1, three colour gradients: 10).
BWD_MIN_INSTR_PER_BLEND = 31


def issue_ceiling(blended: int, ms: float, sms: int, sm_mhz: float, inst=None) -> dict:
    """The backward against its issue ceiling: every blended pair's method
    minimum on fully used lanes, at one warp instruction a cycle on each of
    the SMs' four schedulers.  inst: the kernel's warp instructions per
    launch from an ncu record of the current source (None if stale)."""
    rate = sms * 4 * sm_mhz * 1e6
    model = blended * BWD_MIN_INSTR_PER_BLEND / 32.0 / rate
    out = {"bound": "issue", "blended_px_splat": blended,
           "min_thread_instructions_per_blend": BWD_MIN_INSTR_PER_BLEND,
           "peak": "%d SMs x 4 schedulers x %.0f MHz (median SM clock under load), one warp "
                   "instruction a cycle each" % (sms, sm_mhz),
           "model_ms": model * 1e3, "frac": model / (ms * 1e-3)}
    if inst:
        out["warp_instructions_per_launch"] = inst
        out["thread_instructions_per_blend"] = 32.0 * inst / max(blended, 1)
        out["issue_frac_if_every_cycle_issued"] = (inst / rate) / (ms * 1e-3)
    return out


def smem_ceiling(ms: float, sms: int, sm_mhz: float, rec) -> dict:
    """The backward's shared-memory traffic against the wavefront peak (one
    128-byte wavefront a cycle per SM): the design's own shared loads and
    stores, counted by ncu on the current source (rec: the committed
    record, None if stale), per launch over the live CUDA-event duration."""
    out = {"bound": "shared-memory wavefronts (this kernel's own traffic, ncu)",
           "peak": "%d SMs x one wavefront a cycle x %.0f MHz (median SM clock under load)"
                   % (sms, sm_mhz)}
    wf = (rec or {}).get("smem_wavefronts_per_launch")
    if not wf:
        out["wavefronts_per_launch"] = None
        return out
    rate = sms * sm_mhz * 1e6
    out.update({"wavefronts_per_launch": wf, "model_ms": wf / rate * 1e3,
                "frac": (wf / rate) / (ms * 1e-3)})
    return out


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return {}


def measure_projection(ss, dev, flush, steps: int, hbm: float, hbm_src: str) -> dict:
    """The projection forward and backward on the 2M-splat, degree-3 scene at
    1237x822, each call timed alone with CUDA events after an L2 flush."""
    import torch
    from synth.scene3d import make_scene3d
    sc = make_scene3d(13)
    sp = ss.Splats3D.from_numpy(sc, dev)
    cam = ss.camera(sc.cam.R, sc.cam.t, sc.cam.fx, sc.cam.fy, sc.cam.cx, sc.cam.cy, sc.cam.near,
                    sc.cam.blur)
    pr = ss.Projector(sc.n, sc.sh_degree, dev)
    f = lambda a: torch.from_numpy(a).to(dev).contiguous()  # noqa: E731
    gm, gc, gr = f(sc.dmean2d), f(sc.dconic), f(sc.drgb)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        pr.forward(sp, cam)
        pr.backward(sp, cam, gm, gc, gr)
    torch.cuda.synchronize()
    times = {"fwd": [], "bwd": []}
    for k in range(steps):
        for name, call in (("fwd", lambda: pr.forward(sp, cam)),
                           ("bwd", lambda: pr.backward(sp, cam, gm, gc, gr))):
            flush.fill_(float(k))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            times[name].append((e0, e1))
    torch.cuda.synchronize()
    K = (sc.sh_degree + 1) ** 2
    bytes_ = {"fwd": sc.n * (40 + 12 * K + 36), "bwd": sc.n * (40 + 12 * K + 32 + 40 + 12 * K)}
    out = {"workload": sc.name, "splats": sc.n, "sh_degree": sc.sh_degree,
           "culled": int((pr.depth == 0).sum().item())}
    for name in ("fwd", "bwd"):
        ms = statistics.mean(a.elapsed_time(b) for a, b in times[name])
        ach = bytes_[name] / (ms * 1e-3) / 1e9
        out[name] = {"kernel": "k_project_" + name, "ms_per_call": ms,
                     "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                                  "frac": ach / hbm, "algorithmic_bytes": bytes_[name],
                                  "peak_source": hbm_src}}
    out["fwd"]["roofline"]["bytes_model"] = "per splat: mean3 12 + scale 12 + quat 16 + SH 12K " \
        "in, mean2d 8 + conic 12 + depth 4 + rgb 12 out (K = 16)"
    out["bwd"]["roofline"]["bytes_model"] = "per splat: mean3, scale, quat 40 + SH 12K + " \
        "upstream 32 in, 40 + 12K gradients out (K = 16)"
    return out


def measure_ssim(ss, dev, flush, steps: int, hbm: float, hbm_src: str) -> dict:
    """The fused L1 + SSIM loss and gradient on a 3 x 822 x 1237 image pair,
    each call timed alone with CUDA events after an L2 flush."""
    import torch
    from synth.images import IMAGE_WORKLOADS, make_image_pair
    x, y = make_image_pair(22)
    C, H, W = x.shape
    xd, yd = torch.from_numpy(x).to(dev), torch.from_numpy(y).to(dev)
    sl = ss.SsimLoss(C, H, W, 0.2, dev)
    for _ in range(3):
        sl(xd, yd)
    torch.cuda.synchronize()
    ss.ss_profile_collect()
    ss.ss_profile_enable(True)
    ev = []
    stream = torch.cuda.current_stream()
    for k in range(steps):
        flush.fill_(float(k))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        sl(xd, yd)
        e1.record(stream)
        ev.append((e0, e1))
    torch.cuda.synchronize()
    ss.ss_profile_enable(False)
    prof = ss.ss_profile_collect()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    k_ms = prof["k_ssim"][1] / prof["k_ssim"][0]
    nbytes = 12 * C * H * W
    ach = nbytes / (k_ms * 1e-3) / 1e9
    return {"workload": IMAGE_WORKLOADS[22].name, "lambda": 0.2, "ms_per_call": ms,
            "kernels_ms_per_call": {k: v[1] / v[0] for k, v in prof.items()},
            "loss": float(sl.loss[0].item()),
            "roofline": {"kernel": "k_ssim", "bound": "hbm", "achieved": ach, "peak": hbm,
                         "unit": "GB/s", "frac": ach / hbm, "algorithmic_bytes": nbytes,
                         "peak_source": hbm_src,
                         "bytes_model": "per pixel and channel: rendered 4 + target 4 read, "
                                        "gradient 4 written"}}


def measure_distortion(ss, dev, flush, steps: int, workload: int = 6, extra_flags=None,
                       label: str = "accum_weight + distortion") -> dict:
    """The step with an output variant (default: accumulated weight + depth
    distortion) on a 2M-splat scene, as a CUDA graph, L2 flushed before each
    replay; per-kernel times from a second, profiled pass."""
    import torch
    import synth
    sc = synth.make_scene(workload)
    flags = ss.SS_ACCUM_WEIGHT | (ss.SS_DISTORTION if extra_flags is None else extra_flags)
    sp = ss.Splats.from_numpy(sc, dev)
    dL = torch.from_numpy(sc.dL_dimage).to(dev).contiguous()
    dLd = (torch.from_numpy(sc.dL_ddist).to(dev).contiguous()
           if flags & ss.SS_DISTORTION else None)
    r = ss.Rasterizer(sc.W, sc.H, sc.n, int(2.5 * sc.n), flags, bg=sc.bg, device=dev)
    r.step(sp, dL, dL_ddist=dLd)
    g = r.capture(sp, dL, dL_ddist=dLd)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    r.check()
    stream = torch.cuda.current_stream()
    ev = []
    for k in range(steps):
        flush.fill_(float(k))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        ev.append((e0, e1))
    torch.cuda.synchronize()
    ss.ss_profile_collect()
    ss.ss_profile_enable(True)
    for k in range(steps):
        flush.fill_(float(k))
        r.step_async(sp, dL, dL_ddist=dLd)
    torch.cuda.synchronize()
    ss.ss_profile_enable(False)
    prof = ss.ss_profile_collect()
    r.check()
    return {"workload": synth.WORKLOADS[workload].name, "flags": label,
            "ms_per_step": statistics.mean(a.elapsed_time(b) for a, b in ev),
            "kernels_ms_per_call": {k: v[1] / v[0] for k, v in prof.items()}}


def measure_splat_entry_points(ss, dev, flush, steps: int, workload: int = 4) -> dict:
    """The boundary's entry points that take the splats themselves
    (ss_raster_fwd: records computed per batch in the kernel, no blend masks;
    ss_raster_bwd: records rebuilt and blend decisions re-evaluated in its
    workspace) on the 2M-splat scene, each call timed alone with CUDA events
    after an L2 flush; per-kernel times from a second, profiled pass."""
    import torch
    import synth
    sc = synth.make_scene(workload)
    flags = ss.SS_ACCUM_WEIGHT
    sp = ss.Splats.from_numpy(sc, dev)
    dL = torch.from_numpy(sc.dL_dimage).to(dev).contiguous()
    r = ss.Rasterizer(sc.W, sc.H, sc.n, int(2.5 * sc.n), flags, bg=sc.bg, device=dev)
    r.bin_and_sort(sp)
    stream = torch.cuda.current_stream()

    def fwd():
        ss.ss_raster_fwd(sp, r.vals, r.tile_offsets, sc.W, sc.H, r.bg, flags, r.image,
                         r.T_final, r.last_contrib, r.median_depth)

    def bwd():
        ss.ss_raster_bwd(sp, r.vals, r.tile_offsets, sc.W, sc.H, r.bg, flags, r.T_final,
                         r.last_contrib, dL, r.grads, r.accum_weight, r.workspace)

    for _ in range(3):
        fwd()
        bwd()
    torch.cuda.synchronize()
    times = {"fwd": [], "bwd": []}
    for k in range(steps):
        for name, fn in (("fwd", fwd), ("bwd", bwd)):
            flush.fill_(float(k))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            times[name].append((e0, e1))
    torch.cuda.synchronize()
    ss.ss_profile_collect()
    ss.ss_profile_enable(True)
    for k in range(steps):
        flush.fill_(float(k))
        fwd()
        flush.fill_(float(k))
        bwd()
    torch.cuda.synchronize()
    ss.ss_profile_enable(False)
    prof = ss.ss_profile_collect()
    st = ss.ss_sort_status(r.workspace)
    if st != 0:
        raise RuntimeError("ss_raster_bwd reported status %d" % st)
    return {"workload": synth.WORKLOADS[workload].name, "flags": "accum_weight",
            "ss_raster_fwd_ms_per_call": statistics.mean(a.elapsed_time(b) for a, b in times["fwd"]),
            "ss_raster_bwd_ms_per_call": statistics.mean(a.elapsed_time(b) for a, b in times["bwd"]),
            "kernels_ms_per_call": {k: v[1] / v[0] for k, v in prof.items()}}


def blended_pairs(masks, cap: int, n_pairs: int) -> int:
    """(pixel, splat) pairs that blended: the bits set in the forward's blend
    masks ([8][cap] words, the first n_pairs of each row in use)."""
    import torch
    lut = torch.tensor([bin(i).count("1") for i in range(256)], dtype=torch.int64,
                       device=masks.device)
    m = masks.view(8, cap)
    return sum(int(lut[m[b, :n_pairs].contiguous().view(torch.uint8).long()].sum().item())
               for b in range(8))


def sort_passes(counters, tiles: int) -> int:
    """Radix passes the device-count sort runs: 8-bit digits of the key
    (tile, depth bits - lo) over the depth range the binning recorded
    (counters [2] / [3]), as the library maps it."""
    tb = max(0, (int(tiles) - 1).bit_length())
    full = (32 + tb + 7) // 8
    lo64, hi64 = int(counters[2]), int(counters[3])
    if not (lo64 <= hi64 <= 0xffffffff):
        return full
    lo = lo64 & 0xffff0000
    db = max(16, (hi64 - lo).bit_length())
    return min(full, (db + tb + 7) // 8)


def kernel_rooflines(kernels: dict, steps: int, n: int, P: int, HW: int, cand: int, active: int,
                     blended: int, hbm: float, hbm_src: str, red_rate: float, accum: bool,
                     sms: int, sm_mhz: float, passes: int = None) -> dict:
    """Every kernel of the step against its roofline, with the per-unit
    algorithmic figures of the path's scope table: HBM bytes for the binning
    and the sort; HBM bytes, L2 reductions and the plain-ALU term (FP32 + MUFU
    instructions at SMs x 128 lanes x the SM clock under load) for the
    rasterizers."""
    def per_call(*names):
        return sum(kernels[k]["ms_total"] for k in names if k in kernels) / steps

    def hbm_row(nbytes, ms, model):
        ach = nbytes / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "algorithmic_bytes": nbytes, "bytes_model": model,
                "ms_per_call": ms, "achieved": ach, "peak": hbm, "unit": "GB/s",
                "frac": ach / hbm, "peak_source": hbm_src}

    lanes = sms * 128 * sm_mhz * 1e6          # FP32 lane-instructions per second

    def alu_row(evals, per_eval, ms, what):
        t = evals * per_eval / lanes
        return {"bound": "alu", "evaluations": evals, "instructions_per_evaluation": per_eval,
                "what": what, "model_ms": t * 1e3, "frac": t / (ms * 1e-3),
                "peak": "%d SMs x 128 FP32 lanes x %.0f MHz (median SM clock under load)" % (
                    sms, sm_mhz)}

    if passes is None:
        passes = kernels.get("k_sort_pass", {}).get("launches", 0) // max(1, steps)
    out = {
        "k_emit_pairs": hbm_row(28 * n + 12 * P, per_call("k_emit_pairs"),
                                "28 B/splat read + 12 B/pair written"),
        "sort (hist, passes, final, ties)": hbm_row(
            (24 * passes + 8 + 8) * P,
            per_call("k_sort_hist", "k_sort_pass", "k_sort_final", "k_sort_ties"),
            "8 B/pair histogram read + 24 B/pair per pass x %d passes run + 8 B/pair offsets" % passes),
    }
    fwd_ms = per_call("k_raster_fwd")
    out["k_raster_fwd"] = {
        "hbm": hbm_row(40 * P + 20 * HW, fwd_ms, "40 B/pair gather + 20 B/pixel written"),
        "alu": alu_row(cand, 16, fwd_ms, "every candidate (pixel, splat) of every tile list, "
                                         "~15 FP32 + 1 MUFU each"),
    }
    bwd_ms = per_call("k_raster_bwd")
    nat = (10 if accum else 9) * P
    out["k_raster_bwd"] = {
        "hbm": hbm_row(40 * P + 20 * HW + (36 + (8 if accum else 0)) * n, bwd_ms,
                       "40 B/pair + 20 B/pixel + %d B/splat" % (36 + (8 if accum else 0))),
        "l2_atomic": {"bound": "l2_atomic", "atomics": nat, "model_ms": nat / red_rate * 1e3,
                      "frac": (nat / red_rate) / (bwd_ms * 1e-3), "peak": red_rate,
                      "unit": "atomic/s"},
        "alu_active": alu_row(active, 47, bwd_ms, "every list entry up to each pixel's last "
                                                  "blended splat (sum of last_contrib), ~45 FP32 "
                                                  "+ 2 MUFU each: a replay without blend masks"),
        "alu_blended": alu_row(blended, 47, bwd_ms, "only the (pixel, splat) pairs that "
                                                    "blended, ~45 FP32 + 2 MUFU each"),
    }
    return out


def run_ours(args, rank: int, world: int, dist):
    import torch
    try:
        import gaussian_splatting_differentiable_gb300 as ss
    except ImportError:
        import __graft_entry__
        __graft_entry__.build()
        import gaussian_splatting_differentiable_gb300 as ss
    import synth

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    scene = synth.make_scene(args.workload)
    wl = synth.WORKLOADS[args.workload]
    flags = (ss.SS_ACCUM_WEIGHT if scene.accum_weight else 0) | \
        (ss.SS_MEDIAN_DEPTH if scene.median_depth else 0)
    sp = ss.Splats.from_numpy(scene, dev)
    dL = torch.from_numpy(scene.dL_dimage).to(dev).contiguous()
    r = ss.Rasterizer(scene.W, scene.H, scene.n, int(2.5 * scene.n), flags, bg=scene.bg,
                      device=dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    r.step(sp, dL)                      # sizes the pair buffers (the one host read)
    for _ in range(args.warmup):
        r.step_async(sp, dL)
    torch.cuda.synchronize()
    r.check()
    offs = r.tile_offsets.cpu().numpy().view(np.uint32)
    cand = candidate_pairs(offs, scene.W, scene.H)
    active = int(r.last_contrib.sum().item())
    P = r.n_pairs

    # The step as one CUDA graph: bin -> sort on the device-side pair count ->
    # forward -> backward, no host synchronisation inside.
    graph = r.capture(sp, dL)
    graph.replay()
    r.check()
    torch.cuda.synchronize()
    blended = blended_pairs(r.blend_masks, r.capacity, P)   # the graph's masks: rows of `capacity`
    n_tiles = ((scene.W + 15) // 16) * ((scene.H + 15) // 16)
    passes_run = sort_passes(r.counters.cpu().numpy().view(np.uint64), n_tiles)

    # --- device-resident timed region (headline): graph replays
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark(True)
    wall0 = time.perf_counter()
    for k in range(args.steps):
        flush.fill_(float(k))           # > L2: every step starts cold
        ev[k][0].record(stream)
        graph.replay()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    wall1 = time.perf_counter()
    if dist:
        dist.barrier()
    clocks.mark(False)
    r.check()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = statistics.mean(step_ms)

    # --- per-kernel timed region: the same step launched without the graph,
    # every kernel bracketed by CUDA events on its stream (SS_PROFILE)
    ss.ss_profile_collect()
    ss.ss_profile_enable(True)
    torch.cuda.synchronize()
    synced_ms = []
    for k in range(args.steps):
        flush.fill_(float(k))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        r.step_async(sp, dL)
        e1.record(stream)
        synced_ms.append((e0, e1))
    torch.cuda.synchronize()
    clocks.mark(False)
    ss.ss_profile_enable(False)
    prof = ss.ss_profile_collect()
    clk = clocks.stop()
    nograph_ms = statistics.mean(a.elapsed_time(b) for a, b in synced_ms)
    print("step ms (graph): mean %.4f min %.4f max %.4f; without graph %.4f; kernels %s" % (
        ms, min(step_ms), max(step_ms), nograph_ms, prof), file=sys.stderr, flush=True)
    if not prof:
        raise RuntimeError("SS_PROFILE recorded no kernel launches")
    ms = max_over_ranks(ms, dist, dev)
    value = job_value(world, cand, ms)
    launches = sum(c for (c, _, _, _) in prof.values())   # per-kernel region; same per graph replay

    kernels = {k: {"launches": c, "ms_per_call": tot / c, "ms_total": tot, "min_ms": mn,
                   "max_ms": mx} for k, (c, tot, mn, mx) in prof.items()}
    stages = {
        "tile isect (bin+sort)": sum(v["ms_total"] for k, v in kernels.items()
                                     if k.startswith(("k_emit", "k_sort"))) / args.steps,
        "raster fwd": kernels.get("k_raster_fwd", {}).get("ms_total", 0.0) / args.steps,
        "raster bwd": sum(v["ms_total"] for k, v in kernels.items()
                          if k in ("k_grad_zero", "k_raster_bwd", "k_grad_final", "k_bwd_zero",
                                   "k_accum_final")) / args.steps,
    }
    k_total = sum(v["ms_total"] for v in kernels.values())
    dom = max(kernels, key=lambda k: kernels[k]["ms_total"])
    for v in kernels.values():
        v["share"] = v["ms_total"] / k_total

    # --- roofline of the backward kernel (and of the dominant kernel)
    peaks = measured_peaks()
    hbm = peaks.get("hbm_gbs")
    hbm_src = "measured" if hbm else "fallback"
    hbm = hbm or 6800.0
    HW = scene.W * scene.H
    bwd_bytes = 40 * P + 20 * HW + (36 + (8 if scene.accum_weight else 0)) * scene.n
    bwd_ms = kernels["k_raster_bwd"]["ms_per_call"]
    achieved = bwd_bytes / (bwd_ms * 1e-3) / 1e9
    # L2 atomic throughput: distinct-address float reductions
    probe = torch.zeros(64 << 20, dtype=torch.float32, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ss.ss_probe_red_f32(probe, 1)
    torch.cuda.synchronize()
    rounds = 4
    e0.record(stream)
    ss.ss_probe_red_f32(probe, rounds)
    e1.record(stream)
    torch.cuda.synchronize()
    red_rate = probe.numel() * rounds / (e0.elapsed_time(e1) * 1e-3)
    del probe
    n_atomics = (10 if scene.accum_weight else 9) * P
    t_atom = n_atomics / red_rate
    t_hbm = bwd_bytes / (hbm * 1e9)
    roofline = {"kernel": "k_raster_bwd", "bound": "hbm", "achieved": achieved, "peak": hbm,
                "unit": "GB/s", "frac": achieved / hbm, "traffic": recorded_traffic("k_raster_bwd", wl.name),
                "peak_source": hbm_src + " (MEASURED_PEAKS.json hbm_gbs, copy test)",
                "algorithmic_bytes": bwd_bytes,
                "bytes_model": "40 B/pair (index + 36 B splat gather) + 20 B/pixel "
                               "(dL 12, T 4, last 4) + %d B/splat (gradients%s)" % (
                                   36 + (8 if scene.accum_weight else 0),
                                   " + 8 B fixed-point weight" if scene.accum_weight else "")}
    roofline_atomic = {"kernel": "k_raster_bwd", "bound": "l2_atomic",
                       "achieved": n_atomics / (bwd_ms * 1e-3), "peak": red_rate, "unit": "atomic/s",
                       "frac": (n_atomics / (bwd_ms * 1e-3)) / red_rate,
                       "count_model": "%d per (splat, tile) pair = method minimum" % (
                           10 if scene.accum_weight else 9),
                       "peak_source": "measured here: red.global.add.f32, 64M distinct addresses"}
    hbm_atomic_frac = max(t_hbm, t_atom) / (bwd_ms * 1e-3)

    # --- the next rows of the path, each timed on its own workload
    next_rows = {}
    if not args.no_next:
        next_rows["f1_projection"] = measure_projection(ss, dev, flush, args.steps, hbm,
                                                        hbm_src + " (MEASURED_PEAKS.json hbm_gbs)")
        next_rows["f4_ssim"] = measure_ssim(ss, dev, flush, args.steps, hbm,
                                            hbm_src + " (MEASURED_PEAKS.json hbm_gbs)")
        next_rows["f2_distortion"] = measure_distortion(ss, dev, flush, args.steps)
        next_rows["f3_weight_stats"] = measure_distortion(
            ss, dev, flush, args.steps, workload=4, extra_flags=ss.SS_WEIGHT_STATS,
            label="accum_weight + weight statistics (max blend weight, blending-pixel count)")
        # the dense-cluster scene (30 % of the splats in four blobs: tiles of up
        # to ~14k pairs), with every optional output of the default path on
        next_rows["dense_blobs"] = measure_distortion(
            ss, dev, flush, args.steps, workload=5, extra_flags=ss.SS_MEDIAN_DEPTH,
            label="accum_weight + median depth, 30 % of the splats in four dense blobs")
        # the boundary's splat-taking forms (not the training step's path)
        next_rows["b_splat_entry_points"] = measure_splat_entry_points(ss, dev, flush, args.steps)

    # --- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        host_in = {k: torch.from_numpy(getattr(scene, k)).pin_memory()
                   for k in ("mean2d", "conic", "opacity", "rgb", "depth")}
        host_dL = torch.from_numpy(scene.dL_dimage).pin_memory()
        dev_in = ss.Splats(**{k: torch.empty_like(v, device=dev) for k, v in host_in.items()})
        dev_dL = torch.empty_like(host_dL, device=dev)
        outs = [r.image, *r.grads.values()] + ([r.accum_weight] if r.accum_weight is not None else [])
        host_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
        bi = sum(v.numel() * v.element_size() for v in host_in.values()) + \
            host_dL.numel() * host_dL.element_size()
        bo = sum(o.numel() * o.element_size() for o in host_out)
        n_e2e = max(3, min(args.steps, 20))

        e2e_graph = r.capture(dev_in, dev_dL)

        def e2e_step():
            for k, v in host_in.items():
                getattr(dev_in, k).copy_(v, non_blocking=True)
            dev_dL.copy_(host_dL, non_blocking=True)
            e2e_graph.replay()
            for h, o in zip(host_out, outs):
                h.copy_(o, non_blocking=True)
            torch.cuda.synchronize()
        e2e_step()
        e2e_ms = []
        for _ in range(n_e2e):
            flush.fill_(0.0)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            e2e_step()
            e2e_ms.append((time.perf_counter() - t0) * 1e3)
        em = statistics.mean(e2e_ms)
        em = max_over_ranks(em, dist, dev)
        r.check()
        serial = {"value": job_value(world, cand, em), "ms_per_step": em, "steps": n_e2e,
                  "how": "one step at a time: pinned host inputs -> device, the step's CUDA "
                         "graph, gradients + image + weights -> pinned host, synchronize; L2 "
                         "flushed before each step; wall clock"}

        # The same through ss.StepPipeline: step k's inputs go in while step
        # k-1 computes and its results come out while step k+1 computes (two
        # buffer sets, two copy streams).  Every step copies all of its inputs
        # in and all of its results out; wall clock over n_pipe steps.
        pipe = ss.StepPipeline(scene.W, scene.H, scene.n, flags, host_in, host_dL, bg=scene.bg,
                               device=dev, capacity=r.capacity)
        host_outs = [pipe.host_output_buffers(), pipe.host_output_buffers()]
        pipe.run(4, host_in, host_dL, host_outs)         # warm-up
        pipe.check()
        n_pipe = max(8, min(4 * args.steps, 80))
        runs = []
        for _ in range(3):   # the median of three wall-clock runs (the host is shared)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            pipe.run(n_pipe, host_in, host_dL, host_outs)
            runs.append((time.perf_counter() - t0) * 1e3 / n_pipe)
        pm = sorted(runs)[1]
        pipe.check()
        pm = max_over_ranks(pm, dist, dev)
        e2e = {"value": job_value(world, cand, pm), "unit": UNIT, "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": bo, "ms_per_step": pm, "steps": n_pipe,
               "runs_ms_per_step": runs,
               "how": "ss.StepPipeline: every step copies its inputs from pinned host memory and "
                      "its image, gradients and weights back to pinned host memory; copies of "
                      "one step overlap the compute of its neighbours (two buffer sets); no L2 "
                      "flush (each step's working set, ~0.5 GB, exceeds the 129 MB L2, and the "
                      "two sets alternate); wall clock over all steps of a run, the median "
                      "of three runs",
               "serial": serial}
        del pipe

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        threads = oracle.default_threads()
        pieces, det = oracle_pieces(scene, 1, threads)
        single = oracle_single_core_rate(scene, 64)
        cpu = {"value": det["candidates"] / sum(pieces), "unit": UNIT, "cores": threads,
               "kind": "oracle",
               "sample": "one whole step of the scene (bin + sort single-threaded, forward + "
                         "backward of every tile tile-parallel on %d threads): %.1f s" % (
                             threads, sum(pieces)),
               "host": cpu_description(), "single_core": single}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "W": scene.W, "H": scene.H, "splats": scene.n,
                   "pairs": P, "candidate_splat_px": cand, "active_px_splat": active,
                   "blended_px_splat": blended,
                   "flags": {"accum_weight": scene.accum_weight, "median_depth": scene.median_depth},
                   "l2": "256 MB buffer written between timed steps (L2 is 129 MB)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "ms_per_step_without_graph": nograph_ms,
        "rasterize_bwd_ms_per_call": stages["raster bwd"],
        "rasterize_bwd_pairs_per_s": cand / (stages["raster bwd"] * 1e-3),
        "k_raster_bwd_ms_per_call": bwd_ms,
        "stages_ms_per_step": stages,
        "kernels": kernels, "dominant_kernel": dom,
        "roofline": roofline, "roofline_atomic": roofline_atomic,
        "bwd_hbm_atomic_roofline_frac": hbm_atomic_frac,
        "roofline_issue": issue_ceiling(
            blended, bwd_ms, torch.cuda.get_device_properties(dev).multi_processor_count,
            clk.get("sm_mhz") or clk.get("sm_max_mhz") or 2070.0,
            (recorded_counters("k_raster_bwd", wl.name) or {}).get("inst_executed_per_launch")),
        "roofline_smem": smem_ceiling(
            bwd_ms, torch.cuda.get_device_properties(dev).multi_processor_count,
            clk.get("sm_mhz") or clk.get("sm_max_mhz") or 2070.0,
            recorded_counters("k_raster_bwd", wl.name)),
        "kernel_rooflines": kernel_rooflines(
            kernels, args.steps, scene.n, P, HW, cand, active, blended, hbm,
            hbm_src + " (MEASURED_PEAKS.json hbm_gbs)", red_rate, scene.accum_weight,
            torch.cuda.get_device_properties(dev).multi_processor_count,
            clk.get("sm_mhz") or clk.get("sm_max_mhz") or 2070.0, passes_run),
        "sort_passes_run": passes_run,
        "l2_red_f32_per_s": red_rate,
        "gpu_launches": launches,
        "next_rows": next_rows,
        "e2e": e2e, "cpu_baseline": cpu, "clocks": clk,
        "wall_ms_per_step": (wall1 - wall0) * 1e3 / args.steps,
    }
    print(json.dumps(line), flush=True)


def run_only(args):
    """One leg of the next rows on its own (a few GB on the device), for ncu."""
    import torch
    try:
        import gaussian_splatting_differentiable_gb300 as ss
    except ImportError:
        import __graft_entry__
        __graft_entry__.build()
        import gaussian_splatting_differentiable_gb300 as ss
    dev = torch.device("cuda", 0)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    peaks = measured_peaks()
    hbm = peaks.get("hbm_gbs") or 6800.0
    src = ("measured" if peaks.get("hbm_gbs") else "fallback") + " (MEASURED_PEAKS.json hbm_gbs)"
    if args.only == "projection":
        out = measure_projection(ss, dev, flush, args.steps, hbm, src)
    elif args.only == "ssim":
        out = measure_ssim(ss, dev, flush, args.steps, hbm, src)
    else:
        out = measure_distortion(ss, dev, flush, args.steps)
    print(json.dumps({"only": args.only, **out}), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        dist = tdist
    if args.only:
        run_only(args)
        return
    try:
        run_ours(args, rank, world, dist)
    finally:
        if dist:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
