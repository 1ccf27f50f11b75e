"""Tile-based differentiable rasterization of projected 2D Gaussian splats on GB300.

The compute path is libss.so (hand-written CUDA for sm_103a behind the C ABI
of include/ss.h, include/ss_project.h and include/ss_ssim.h).  This module is its thin Python binding: each ss_* function
here has the C function's name and arguments and only marshals torch tensors
(device memory) and streams into pointers.  PyTorch provides memory and
streams; every step of the path runs in the library's kernels.  There is no
fallback: importing this package without the built library raises
ImportError.
"""
from __future__ import annotations

import ctypes
import dataclasses

import torch

from . import _lib
from ._lib import (SS_ACCUM_WEIGHT, SS_DISTORTION, SS_ERR_CAPACITY, SS_ERR_DEVICE,  # noqa: F401
                   SS_ERR_TIMEOUT, SS_MEDIAN_DEPTH, SS_OK, SS_RECORDS_CLEARED, SS_WEIGHT_STATS,
                   STATUS_NAMES, SsGrads, SsSplats)

_L = _lib.load()
TILE = 16


class SSError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = _L.ss_last_error().decode(errors="replace")
        super().__init__("%s: %s: %s" % (where, STATUS_NAMES.get(status, status), msg))
        self.status = status


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, where: str):
    if st != SS_OK:
        raise SSError(st, where)


def _f32_host3(bg):
    if bg is None:
        return None
    return (ctypes.c_float * 3)(*[float(x) for x in bg])


@dataclasses.dataclass
class Splats:
    """Device SoA splats (float32, contiguous): mean2d [n,2], conic [n,3],
    opacity [n], rgb [n,3], depth [n]."""
    mean2d: torch.Tensor
    conic: torch.Tensor
    opacity: torch.Tensor
    rgb: torch.Tensor
    depth: torch.Tensor

    @property
    def n(self) -> int:
        return int(self.opacity.shape[0])

    def c(self) -> SsSplats:
        for k in ("mean2d", "conic", "opacity", "rgb", "depth"):
            t = getattr(self, k)
            if t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda:
                raise ValueError("Splats.%s must be a contiguous float32 CUDA tensor" % k)
        return SsSplats(_ptr(self.mean2d), _ptr(self.conic), _ptr(self.opacity), _ptr(self.rgb),
                        _ptr(self.depth), self.n)

    @staticmethod
    def from_numpy(scene, device="cuda") -> "Splats":
        f = lambda a: torch.from_numpy(a).to(device=device, dtype=torch.float32).contiguous()  # noqa
        return Splats(f(scene.mean2d), f(scene.conic), f(scene.opacity), f(scene.rgb),
                      f(scene.depth))


# ------------------------------------------------------------------ C ABI

def ss_abi_version() -> int:
    return int(_L.ss_abi_version())


def ss_constants() -> dict:
    buf = (ctypes.c_float * 4)()
    _L.ss_constants(buf)
    return {"alpha_min": buf[0], "alpha_max": buf[1], "T_eps": buf[2], "tile": int(buf[3])}


def ss_last_error() -> str:
    return _L.ss_last_error().decode(errors="replace")


def ss_workspace_bytes(n_splats: int, n_pairs: int, W: int, H: int) -> int:
    return int(_L.ss_workspace_bytes(n_splats, n_pairs, W, H))


COUNTER_WORDS = 4   # ss_bin_tiles' uint64 counters: pairs, culled, depth-bit range


def _counters(counters):
    """The counters tensor's pointer, after checking that it holds the four
    64-bit words the library writes (a plain pointer crosses the C ABI)."""
    if isinstance(counters, torch.Tensor) and counters.numel() * counters.element_size() < 8 * COUNTER_WORDS:
        raise ValueError("counters must hold %d 64-bit words (got %d bytes)"
                         % (COUNTER_WORDS, counters.numel() * counters.element_size()))
    return _ptr(counters)


def ss_record_bytes(n_splats: int) -> int:
    return int(_L.ss_record_bytes(n_splats))


def ss_bin_tiles(splats: Splats, W: int, H: int, keys, vals, capacity: int, counters, records,
                 stream=None) -> None:
    s = splats.c()
    _check(_L.ss_bin_tiles(ctypes.byref(s), W, H, _ptr(keys), _ptr(vals), capacity,
                           _counters(counters), _ptr(records), _stream(stream)), "ss_bin_tiles")


def ss_pair_count(counters, capacity: int, stream=None):
    """(status, pairs needed, culled); status is SS_OK or SS_ERR_CAPACITY."""
    pairs, culled = ctypes.c_int64(0), ctypes.c_int64(0)
    st = _L.ss_pair_count(_counters(counters), capacity, ctypes.byref(pairs), ctypes.byref(culled),
                          _stream(stream))
    if st not in (SS_OK, SS_ERR_CAPACITY):
        raise SSError(st, "ss_pair_count")
    return st, pairs.value, culled.value


def ss_sort_pairs(keys, vals, n_pairs: int, W: int, H: int, tile_offsets, workspace,
                  stream=None) -> None:
    _check(_L.ss_sort_pairs(_ptr(keys), _ptr(vals), n_pairs, W, H, _ptr(tile_offsets),
                            _ptr(workspace), workspace.numel() * workspace.element_size(),
                            _stream(stream)), "ss_sort_pairs")


def ss_sort_pairs_dev(keys, vals, counters, capacity: int, W: int, H: int, tile_offsets,
                      workspace, stream=None) -> None:
    _check(_L.ss_sort_pairs_dev(_ptr(keys), _ptr(vals), _counters(counters), capacity, W, H,
                                _ptr(tile_offsets), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream)),
           "ss_sort_pairs_dev")


def ss_sort_status(workspace, stream=None) -> int:
    return int(_L.ss_sort_status(_ptr(workspace), _stream(stream)))


def ss_raster_fwd(splats: Splats, vals, tile_offsets, W: int, H: int, bg, flags: int, image,
                  T_final, last_contrib, median_depth=None, stream=None) -> None:
    """The forward from the splats themselves (no records, no blend masks)."""
    s = splats.c()
    _check(_L.ss_raster_fwd(ctypes.byref(s), _ptr(vals), _ptr(tile_offsets), W, H,
                            _f32_host3(bg), flags, _ptr(image), _ptr(T_final), _ptr(last_contrib),
                            _ptr(median_depth), _stream(stream)), "ss_raster_fwd")


def ss_raster_fwd_records(records, n_splats: int, vals, tile_offsets, n_pairs: int, W: int,
                          H: int, bg, flags: int, image, T_final, last_contrib, median_depth,
                          blend_masks, max_weight=None, blend_count=None, distortion=None,
                          dist_totals=None, stream=None, bwd_workspace=None) -> None:
    """bwd_workspace: the workspace of the following ss_raster_bwd_records,
    whose gradient records the forward then clears (pass SS_RECORDS_CLEARED
    to that call; nothing may write the workspace in between)."""
    nbytes = 0 if bwd_workspace is None else bwd_workspace.numel() * bwd_workspace.element_size()
    _check(_L.ss_raster_fwd_records(_ptr(records), n_splats, _ptr(vals), _ptr(tile_offsets),
                                    n_pairs, W, H, _f32_host3(bg), flags, _ptr(image),
                                    _ptr(T_final), _ptr(last_contrib), _ptr(median_depth),
                                    _ptr(blend_masks), _ptr(max_weight), _ptr(blend_count),
                                    _ptr(distortion), _ptr(dist_totals), _ptr(bwd_workspace),
                                    nbytes, _stream(stream)), "ss_raster_fwd_records")


def _grads_struct(grads: dict) -> SsGrads:
    return SsGrads(_ptr(grads["dmean2d"]), _ptr(grads["dconic"]), _ptr(grads["dopacity"]),
                   _ptr(grads["drgb"]), _ptr(grads.get("ddepth")))


def ss_raster_bwd(splats: Splats, vals, tile_offsets, W: int, H: int, bg, flags: int, T_final,
                  last_contrib, dL_dimage, grads: dict, accum_weight, workspace,
                  stream=None) -> None:
    """The backward from the splats themselves: records and blend decisions
    rebuilt in the workspace (ss_workspace_bytes(n, pairs, W, H) bytes)."""
    s = splats.c()
    g = _grads_struct(grads)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_L.ss_raster_bwd(ctypes.byref(s), _ptr(vals), _ptr(tile_offsets), W, H,
                            _f32_host3(bg), flags, _ptr(T_final), _ptr(last_contrib),
                            _ptr(dL_dimage), ctypes.byref(g), _ptr(accum_weight),
                            _ptr(workspace), nbytes, _stream(stream)), "ss_raster_bwd")


def ss_raster_bwd_records(records, n_splats: int, vals, tile_offsets, n_pairs: int, W: int,
                          H: int, bg, flags: int, T_final, last_contrib, blend_masks, dL_dimage,
                          grads: dict, accum_weight, workspace, stream=None, dist_totals=None,
                          dL_ddist=None) -> None:
    """blend_masks may be None: the decisions are then re-evaluated into the
    workspace."""
    g = _grads_struct(grads)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_L.ss_raster_bwd_records(_ptr(records), n_splats, _ptr(vals), _ptr(tile_offsets),
                                    n_pairs, W, H, _f32_host3(bg), flags, _ptr(T_final),
                                    _ptr(last_contrib), _ptr(blend_masks), _ptr(dL_dimage),
                                    _ptr(dist_totals), _ptr(dL_ddist), ctypes.byref(g),
                                    _ptr(accum_weight), _ptr(workspace), nbytes,
                                    _stream(stream)), "ss_raster_bwd_records")


def ss_raster_bwd_noalloc(records, n_splats: int, vals, tile_offsets, n_pairs: int, W: int,
                          H: int, bg, flags: int, T_final, last_contrib, blend_masks, dL_dimage,
                          grads: dict, accum_weight, stream=None) -> None:
    """ss_raster_bwd_records for callers that cannot allocate: no workspace argument;
    the weight scratch is a fixed array inside the library (at most 2,097,152
    splats; concurrent calls race on it)."""
    g = _grads_struct(grads)
    _check(_L.ss_raster_bwd_noalloc(_ptr(records), n_splats, _ptr(vals), _ptr(tile_offsets),
                                    n_pairs, W, H, _f32_host3(bg), flags, _ptr(T_final),
                                    _ptr(last_contrib), _ptr(blend_masks), _ptr(dL_dimage),
                                    ctypes.byref(g), _ptr(accum_weight),
                                    _stream(stream)), "ss_raster_bwd_noalloc")


def ss_profile_enable(on: bool) -> None:
    _L.ss_profile_enable(1 if on else 0)


def ss_profile_collect() -> dict:
    """{kernel name: (launches, total_ms, min_ms, max_ms)} since the last collect."""
    buf = ctypes.create_string_buffer(1 << 20)   # one line per kernel name
    _L.ss_profile_collect(buf, len(buf))
    out = {}
    for line in buf.value.decode().splitlines():
        name, cnt, tot, mn, mx = line.split()
        out[name] = (int(cnt), float(tot), float(mn), float(mx))
    return out


def ss_debug_bounds_enabled() -> bool:
    return bool(_L.ss_debug_bounds_enabled())


def ss_debug_status(stream=None) -> int:
    """SS_OK, or SS_ERR_DEVICE if a device-side bounds check failed since the
    last call (only the SS_DEBUG_BOUNDS build checks; see ss_last_error())."""
    return int(_L.ss_debug_status(_stream(stream)))


def ss_probe_red_f32(buf, rounds: int, stream=None) -> None:
    _check(_L.ss_probe_red_f32(_ptr(buf), buf.numel(), rounds, _stream(stream)),
           "ss_probe_red_f32")


def ss_test_sort_wait_timeout(workspace, stream=None) -> None:
    _check(_L.ss_test_sort_wait_timeout(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _stream(stream)), "ss_test_sort_wait_timeout")


# ------------------------------------------------------------------ projection (ss_project.h)

@dataclasses.dataclass
class Splats3D:
    """Device 3D splats (float32, contiguous): mean3 [n,3], scale [n,3],
    quat [n,4] (w, x, y, z), sh [K,3,n] coefficient-major, K = (degree+1)^2."""
    mean3: torch.Tensor
    scale: torch.Tensor
    quat: torch.Tensor
    sh: torch.Tensor
    sh_degree: int

    @property
    def n(self) -> int:
        return int(self.mean3.shape[0])

    def c(self) -> _lib.SsSplats3d:
        for k in ("mean3", "scale", "quat", "sh"):
            t = getattr(self, k)
            if t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda:
                raise ValueError("Splats3D.%s must be a contiguous float32 CUDA tensor" % k)
        return _lib.SsSplats3d(_ptr(self.mean3), _ptr(self.scale), _ptr(self.quat),
                               _ptr(self.sh), self.n, self.sh_degree)

    @staticmethod
    def from_numpy(scene, device="cuda") -> "Splats3D":
        f = lambda a: torch.from_numpy(a).to(device=device, dtype=torch.float32).contiguous()  # noqa
        return Splats3D(f(scene.mean3), f(scene.scale), f(scene.quat), f(scene.sh),
                        scene.sh_degree)


def camera(R, t, fx: float, fy: float, cx: float, cy: float, near: float,
           blur: float) -> _lib.SsCamera:
    """The host ss_camera struct (R row-major world-to-camera rotation)."""
    c = _lib.SsCamera()
    for k, v in enumerate([float(x) for row in R for x in row]):
        c.R[k] = v
    for k in range(3):
        c.t[k] = float(t[k])
    c.fx, c.fy, c.cx, c.cy, c.near_z, c.blur = fx, fy, cx, cy, near, blur
    return c


def ss_project_fwd(splats: Splats3D, cam: _lib.SsCamera, mean2d, conic, depth, rgb,
                   stream=None) -> None:
    s = splats.c()
    _check(_L.ss_project_fwd(ctypes.byref(s), ctypes.byref(cam), _ptr(mean2d), _ptr(conic),
                             _ptr(depth), _ptr(rgb), _stream(stream)), "ss_project_fwd")


def ss_project_bwd(splats: Splats3D, cam: _lib.SsCamera, dmean2d, dconic, drgb, grads: dict,
                   stream=None) -> None:
    """grads: dict of device tensors dmean3, dscale, dquat, dsh (overwritten)."""
    s = splats.c()
    g = _lib.SsGrads3d(*[_ptr(grads[k]) for k in ("dmean3", "dscale", "dquat", "dsh")])
    _check(_L.ss_project_bwd(ctypes.byref(s), ctypes.byref(cam), _ptr(dmean2d), _ptr(dconic),
                             _ptr(drgb), ctypes.byref(g), _stream(stream)), "ss_project_bwd")


class Projector:
    """Output and gradient buffers of the projection for n splats; the 2D
    outputs plus a caller's opacity form the rasterizer's Splats."""

    def __init__(self, n: int, sh_degree: int, device="cuda"):
        d = torch.device(device)
        f = lambda *s: torch.empty(*s, dtype=torch.float32, device=d)  # noqa: E731
        K = (sh_degree + 1) ** 2
        self.n, self.sh_degree = n, sh_degree
        self.mean2d, self.conic, self.depth, self.rgb = f(n, 2), f(n, 3), f(n), f(n, 3)
        self.grads = {"dmean3": f(n, 3), "dscale": f(n, 3), "dquat": f(n, 4), "dsh": f(K, 3, n)}

    def forward(self, splats: Splats3D, cam, stream=None) -> None:
        ss_project_fwd(splats, cam, self.mean2d, self.conic, self.depth, self.rgb, stream)

    def backward(self, splats: Splats3D, cam, dmean2d, dconic, drgb, stream=None) -> None:
        ss_project_bwd(splats, cam, dmean2d, dconic, drgb, self.grads, stream)

    def splats2d(self, opacity) -> Splats:
        return Splats(self.mean2d, self.conic, opacity, self.rgb, self.depth)


# ------------------------------------------------------------------ L1 + SSIM loss (ss_ssim.h)

def ss_ssim_workspace_bytes(C: int, H: int, W: int) -> int:
    return int(_L.ss_ssim_workspace_bytes(C, H, W))


def ss_ssim_loss(img, target, lam: float, loss, dL_dimg, workspace, stream=None) -> None:
    """img, target, dL_dimg: [C,H,W] float32 device tensors; loss: float32[3]
    device tensor (loss, mean SSIM, mean |x - y|)."""
    C, H, W = img.shape
    _check(_L.ss_ssim_loss(_ptr(img), _ptr(target), C, H, W, float(lam), _ptr(loss),
                           _ptr(dL_dimg), _ptr(workspace),
                           workspace.numel() * workspace.element_size(), _stream(stream)),
           "ss_ssim_loss")


class SsimLoss:
    """Buffers of ss_ssim_loss for one image size."""

    def __init__(self, C: int, H: int, W: int, lam: float = 0.2, device="cuda"):
        d = torch.device(device)
        self.lam = lam
        self.loss = torch.zeros(3, dtype=torch.float32, device=d)
        self.grad = torch.empty(C, H, W, dtype=torch.float32, device=d)
        nb = max(ss_ssim_workspace_bytes(C, H, W), 16)
        self.workspace = torch.empty((nb + 15) // 16, 2, dtype=torch.float64, device=d)

    def __call__(self, img, target, stream=None) -> torch.Tensor:
        ss_ssim_loss(img, target, self.lam, self.loss, self.grad, self.workspace, stream)
        return self.grad


# ------------------------------------------------------------------ whole path

class Rasterizer:
    """Buffers for one image size and splat count, reused across calls, and
    the call sequence bin -> pair count -> sort -> forward / backward.

    Pair buffers grow (once) when the binning reports more pairs than their
    capacity; nothing else is allocated after construction."""

    def __init__(self, W: int, H: int, n_splats: int, pair_capacity: int, flags: int = 0,
                 bg=None, device="cuda"):
        self.W, self.H, self.n, self.flags = W, H, n_splats, flags
        self.bg = None if bg is None else [float(x) for x in bg]
        self.device = torch.device(device)
        self.tiles = ((W + TILE - 1) // TILE) * ((H + TILE - 1) // TILE)
        d = self.device
        self.counters = torch.zeros(COUNTER_WORDS, dtype=torch.int64, device=d)
        self.records = torch.empty(max(ss_record_bytes(n_splats), 16), dtype=torch.uint8, device=d)
        self.tile_offsets = torch.zeros(self.tiles + 1, dtype=torch.int32, device=d)
        self._alloc_pairs(max(int(pair_capacity), 1))
        self.image = torch.empty(3, H, W, dtype=torch.float32, device=d)
        self.T_final = torch.empty(H, W, dtype=torch.float32, device=d)
        self.last_contrib = torch.empty(H, W, dtype=torch.int32, device=d)
        self.median_depth = (torch.empty(H, W, dtype=torch.float32, device=d)
                             if flags & SS_MEDIAN_DEPTH else None)
        self.grads = {"dmean2d": torch.empty(n_splats, 2, dtype=torch.float32, device=d),
                      "dconic": torch.empty(n_splats, 3, dtype=torch.float32, device=d),
                      "dopacity": torch.empty(n_splats, dtype=torch.float32, device=d),
                      "drgb": torch.empty(n_splats, 3, dtype=torch.float32, device=d)}
        self.accum_weight = (torch.empty(n_splats, dtype=torch.float32, device=d)
                             if flags & SS_ACCUM_WEIGHT else None)
        stats = flags & SS_WEIGHT_STATS
        self.max_weight = torch.empty(n_splats, dtype=torch.float32, device=d) if stats else None
        self.blend_count = torch.empty(n_splats, dtype=torch.int32, device=d) if stats else None
        dist = flags & SS_DISTORTION
        self.distortion = torch.empty(H, W, dtype=torch.float32, device=d) if dist else None
        self.dist_totals = torch.empty(H, W, 4, dtype=torch.float32, device=d) if dist else None
        if dist:
            self.grads["ddepth"] = torch.empty(n_splats, dtype=torch.float32, device=d)
        self.n_pairs = 0
        self.culled = 0
        self._records_cleared = False   # the forward cleared the backward's records since the last sort

    def _alloc_pairs(self, cap: int):
        d = self.device
        self.capacity = cap
        self.keys = torch.empty(cap, dtype=torch.int64, device=d)
        self.vals = torch.empty(cap, dtype=torch.int32, device=d)
        self.blend_masks = torch.empty(8 * cap, dtype=torch.int32, device=d)
        ws = ss_workspace_bytes(self.n, cap, self.W, self.H)
        if ws == 0:
            raise ValueError("sizes out of range")
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=d)

    def bin_and_sort(self, splats: Splats, stream=None) -> int:
        """Tile lists of `splats`; returns the number of pairs (one host sync)."""
        ss_bin_tiles(splats, self.W, self.H, self.keys, self.vals, self.capacity, self.counters,
                     self.records, stream)
        st, pairs, culled = ss_pair_count(self.counters, self.capacity, stream)
        if st == SS_ERR_CAPACITY:
            self._alloc_pairs(int(pairs * 1.25) + 1024)
            ss_bin_tiles(splats, self.W, self.H, self.keys, self.vals, self.capacity,
                         self.counters, self.records, stream)
            st, pairs, culled = ss_pair_count(self.counters, self.capacity, stream)
            _check(st, "ss_pair_count")
        self.n_pairs, self.culled = pairs, culled
        ss_sort_pairs(self.keys, self.vals, pairs, self.W, self.H, self.tile_offsets,
                      self.workspace, stream)
        self._records_cleared = False   # the sort wrote the workspace
        return pairs

    def forward(self, splats: Splats = None, stream=None) -> None:
        """Composite; uses the records written by the last bin_and_sort.  Also
        clears the backward's gradient records in the workspace, so that the
        next backward() skips that pass; bin_and_sort() resets that, but a
        sort called directly on this workspace between forward() and
        backward() must be followed by forward() again."""
        ss_raster_fwd_records(self.records, self.n, self.vals, self.tile_offsets, self.n_pairs,
                              self.W, self.H, self.bg, self.flags, self.image, self.T_final,
                              self.last_contrib, self.median_depth, self.blend_masks,
                              self.max_weight, self.blend_count, self.distortion,
                              self.dist_totals, stream, bwd_workspace=self.workspace)
        self._records_cleared = True

    def backward(self, splats, dL_dimage: torch.Tensor, stream=None, dL_ddist=None) -> None:
        """Gradients; uses the records written by the last bin_and_sort.
        dL_ddist: [H, W] upstream gradient of the distortion (SS_DISTORTION)."""
        flags = self.flags | (SS_RECORDS_CLEARED if self._records_cleared else 0)
        ss_raster_bwd_records(self.records, self.n, self.vals, self.tile_offsets, self.n_pairs,
                              self.W, self.H, self.bg, flags, self.T_final, self.last_contrib,
                              self.blend_masks, dL_dimage, self.grads, self.accum_weight,
                              self.workspace, stream, self.dist_totals, dL_ddist)
        self._records_cleared = False   # the backward's sums are in them now

    def step(self, splats: Splats, dL_dimage: torch.Tensor, stream=None, dL_ddist=None) -> int:
        """One pass of the whole path: bin, sort, forward, backward."""
        n = self.bin_and_sort(splats, stream)
        self.forward(splats, stream)
        self.backward(splats, dL_dimage, stream, dL_ddist)
        return n

    def step_async(self, splats: Splats, dL_dimage: torch.Tensor, stream=None,
                   dL_ddist=None) -> None:
        """bin -> sort -> forward -> backward with the pair count kept on the
        device: no host synchronisation, so the step can be captured in a
        CUDA graph.  The pair buffers must already be large enough (size them
        with one step() first); check() reports an overflow afterwards."""
        ss_bin_tiles(splats, self.W, self.H, self.keys, self.vals, self.capacity, self.counters,
                     self.records, stream)
        ss_sort_pairs_dev(self.keys, self.vals, self.counters, self.capacity, self.W, self.H,
                          self.tile_offsets, self.workspace, stream)
        ss_raster_fwd_records(self.records, self.n, self.vals, self.tile_offsets, self.capacity,
                              self.W, self.H, self.bg, self.flags, self.image, self.T_final,
                              self.last_contrib, self.median_depth, self.blend_masks,
                              self.max_weight, self.blend_count, self.distortion,
                              self.dist_totals, stream, bwd_workspace=self.workspace)
        ss_raster_bwd_records(self.records, self.n, self.vals, self.tile_offsets, self.capacity,
                              self.W, self.H, self.bg, self.flags | SS_RECORDS_CLEARED,
                              self.T_final, self.last_contrib, self.blend_masks, dL_dimage,
                              self.grads, self.accum_weight, self.workspace, stream,
                              self.dist_totals, dL_ddist)

    def check(self, stream=None) -> None:
        """Raise if the last sort reported a device-side problem (capacity
        overflow, look-back timeout, out-of-range key)."""
        _check(ss_sort_status(self.workspace, stream), "sort status")

    def capture(self, splats: Splats, dL_dimage: torch.Tensor,
                dL_ddist=None) -> "torch.cuda.CUDAGraph":
        """A CUDA graph of step_async on these buffers (replay with .replay())."""
        self.step_async(splats, dL_dimage, dL_ddist=dL_ddist)   # first calls set attributes
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step_async(splats, dL_dimage, dL_ddist=dL_ddist)
        return g


class StepPipeline:
    """The whole step (bin, sort, forward, backward) fed from and returned to
    pinned host memory, double-buffered across steps on one GPU.

    Two buffer sets, each a Rasterizer with its own captured CUDA graph and
    device input buffers, and three streams: step k's host-to-device input
    copy runs on one copy stream while step k-1 computes, step k's results
    (image, gradients, accumulated weight) come back on a second copy stream
    while step k+1 computes, and events order each buffer set's copy in,
    compute and copy out.  Every step still copies all of its inputs in and
    all of its results out; the copies overlap the other set's compute.

    The pair buffers must be sized first (the constructor runs one
    synchronous step on the given inputs); check() after run() reports a
    capacity overflow or another device-side problem of the last steps."""

    KEYS = ("mean2d", "conic", "opacity", "rgb", "depth")

    def __init__(self, W: int, H: int, n_splats: int, flags: int, host_splats: dict, host_dL,
                 bg=None, device="cuda", capacity=None):
        d = torch.device(device)
        self.device = d
        cap = capacity if capacity is not None else max(64, 3 * n_splats)
        self.r, self.dev_in, self.dev_dL, self.graphs = [], [], [], []
        for b in range(2):
            r = Rasterizer(W, H, n_splats, cap, flags, bg=bg, device=d)
            sp = Splats(**{k: torch.empty(host_splats[k].shape, dtype=torch.float32, device=d)
                           for k in self.KEYS})
            dL = torch.empty(host_dL.shape, dtype=torch.float32, device=d)
            for k in self.KEYS:
                getattr(sp, k).copy_(host_splats[k])
            dL.copy_(host_dL)
            r.step(sp, dL)                 # sizes the pair buffers (one host read)
            self.r.append(r)
            self.dev_in.append(sp)
            self.dev_dL.append(dL)
        for b in range(2):
            self.graphs.append(self.r[b].capture(self.dev_in[b], self.dev_dL[b]))
        torch.cuda.synchronize()
        self.h2d = torch.cuda.Stream(device=d)
        self.comp = torch.cuda.Stream(device=d)
        self.d2h = torch.cuda.Stream(device=d)
        ev = lambda: [torch.cuda.Event(), torch.cuda.Event()]  # noqa: E731
        self.in_ready, self.computed, self.out_read, self.in_free = ev(), ev(), ev(), ev()
        self.started = [False, False]

    def outputs(self, b: int) -> list:
        r = self.r[b]
        out = [r.image] + [r.grads[k] for k in ("dmean2d", "dconic", "dopacity", "drgb")]
        if r.accum_weight is not None:
            out.append(r.accum_weight)
        return out

    def host_output_buffers(self, pin=True) -> list:
        return [torch.empty(o.shape, dtype=o.dtype, pin_memory=pin) for o in self.outputs(0)]

    def submit(self, k: int, host_splats: dict, host_dL, host_out: list) -> None:
        """Enqueue step k: copy in, compute, copy out (all asynchronous)."""
        b = k & 1
        with torch.cuda.stream(self.h2d):
            if self.started[b]:
                self.h2d.wait_event(self.in_free[b])        # step k-2 has read its inputs
            for key in self.KEYS:
                getattr(self.dev_in[b], key).copy_(host_splats[key], non_blocking=True)
            self.dev_dL[b].copy_(host_dL, non_blocking=True)
            self.in_ready[b].record(self.h2d)
        with torch.cuda.stream(self.comp):
            self.comp.wait_event(self.in_ready[b])
            if self.started[b]:
                self.comp.wait_event(self.out_read[b])      # step k-2's results are out
            self.graphs[b].replay()
            self.computed[b].record(self.comp)
            self.in_free[b].record(self.comp)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(self.computed[b])
            for h, o in zip(host_out, self.outputs(b)):
                h.copy_(o, non_blocking=True)
            self.out_read[b].record(self.d2h)
        self.started[b] = True

    def run(self, steps: int, host_splats: dict, host_dL, host_outs: list) -> None:
        """Enqueue `steps` steps (host_outs: two lists of host output buffers,
        used alternately) and wait for all of them."""
        for k in range(steps):
            self.submit(k, host_splats, host_dL, host_outs[k & 1])
        self.d2h.synchronize()

    def check(self) -> None:
        torch.cuda.synchronize()
        for r in self.r:
            r.check()
