"""The C-ABI library on the host (no GPU): it loads, exports every function
that include/ss.h, ss_project.h and ss_ssim.h declare, reports the oracle's constants, sizes its
workspace, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in ("ss.h", "ss_project.h", "ss_ssim.h")]


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from gaussian_splatting_differentiable_gb300 import _lib
    return _lib.load()


def declared_functions():
    src = "".join(open(h).read() for h in HEADERS)
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ss_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("ss_bin_tiles", "ss_pair_count", "ss_sort_pairs", "ss_raster_fwd", "ss_raster_bwd",
              "ss_workspace_bytes", "ss_last_error", "ss_constants", "ss_project_fwd",
              "ss_project_bwd", "ss_ssim_loss", "ss_ssim_workspace_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from gaussian_splatting_differentiable_gb300 import _lib
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (ss_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)
    assert set(_lib.PROTOTYPES) == set(declared_functions())


def test_constants_match_oracle(lib):
    buf = (ctypes.c_float * 4)()
    lib.ss_constants(buf)
    c = oracle.constants()
    assert buf[0] == np.float32(c["alpha_min"])
    assert buf[1] == np.float32(c["alpha_max"])
    assert buf[2] == np.float32(c["T_eps"])
    assert buf[3] == c["tile"]
    assert lib.ss_abi_version() == 8


def test_workspace_bytes(lib):
    a = lib.ss_workspace_bytes(2_000_000, 5_000_000, 1237, 822)
    assert a >= 5_000_000 * 12 and a % 256 == 0
    assert lib.ss_workspace_bytes(2_000_000, 0, 1237, 822) >= 2_000_000 * 8
    # the backward from the splats builds records (64 B a splat) and blend
    # masks (32 B a pair) after its gradient records (48 B a splat)
    assert a >= 2_000_000 * (48 + 64) + 5_000_000 * 32
    assert lib.ss_workspace_bytes(0, 0, 1, 1) > 0
    assert lib.ss_workspace_bytes(-1, 0, 16, 16) == 0
    assert lib.ss_workspace_bytes(0, 0, 0, 16) == 0
    assert lib.ss_workspace_bytes(0, 1 << 32, 16, 16) == 0
    assert lib.ss_workspace_bytes(0, 0, 40000, 16) == 0


def test_argument_errors_are_reported_before_any_launch(lib):
    from gaussian_splatting_differentiable_gb300._lib import SsSplats, SsGrads
    s = SsSplats(None, None, None, None, None, 10)
    cnt = ctypes.c_void_p(0x1000)
    # image size
    assert lib.ss_bin_tiles(ctypes.byref(s), 0, 16, None, None, 0, cnt, 0x1000, None) == 5
    assert "image" in lib.ss_last_error().decode()
    # NULL splat arrays with n > 0
    assert lib.ss_bin_tiles(ctypes.byref(s), 16, 16, None, None, 0, cnt, 0x1000, None) == 1
    assert lib.ss_bin_tiles(None, 16, 16, None, None, 0, cnt, 0x1000, None) == 1
    # counters NULL; records NULL or unaligned
    s0 = SsSplats(None, None, None, None, None, 0)
    assert lib.ss_bin_tiles(ctypes.byref(s0), 16, 16, None, None, 0, None, None, None) == 1
    sp = SsSplats(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 4)
    assert lib.ss_bin_tiles(ctypes.byref(sp), 16, 16, None, None, 0, cnt, None, None) == 1
    assert lib.ss_bin_tiles(ctypes.byref(sp), 16, 16, None, None, 0, cnt, 0x1008, None) == 1
    assert lib.ss_record_bytes(10) == 640 and lib.ss_record_bytes(-1) == 0
    # sort: too many pairs, NULL offsets, unaligned workspace, small workspace
    assert lib.ss_sort_pairs(None, None, 1 << 32, 16, 16, 0x1000, 0x1000, 1 << 30, None) == 5
    assert lib.ss_sort_pairs(0x1000, 0x1000, 10, 16, 16, None, 0x1000, 1 << 30, None) == 1
    assert lib.ss_sort_pairs(0x1000, 0x1000, 10, 16, 16, 0x1000, 0x1001, 1 << 30, None) == 1
    assert lib.ss_sort_pairs(0x1000, 0x1000, 10, 16, 16, 0x1000, 0x1000, 16, None) == 1
    assert "workspace" in lib.ss_last_error().decode()
    # forward: unknown flags, NULL outputs, median / stats / distortion flag without buffers
    F = lambda *a: lib.ss_raster_fwd_records(*a[:-1], None, 0, a[-1])  # noqa: E731  (no bwd_workspace)
    assert F(None, 0, 0x1000, 0x1000, 0, 16, 16, None, 16, 0x1000, 0x1000, 0x1000, None, 0x1000,
             None, None, None, None, None) == 1
    assert F(None, 0, 0x1000, 0x1000, 0, 16, 16, None, 0, None, 0x1000, 0x1000, None, 0x1000,
             None, None, None, None, None) == 1
    assert F(None, 0, 0x1000, 0x1000, 0, 16, 16, None, 2, 0x1000, 0x1000, 0x1000, None, 0x1000,
             None, None, None, None, None) == 1
    assert F(None, 5, 0x1000, 0x1000, 0, 16, 16, None, 0, 0x1000, 0x1000, 0x1000, None, 0x1000,
             None, None, None, None, None) == 1
    assert F(0x1000, 5, 0x1000, 0x1000, 10, 16, 16, None, 0, 0x1000, 0x1000, 0x1000, None, None,
             None, None, None, None, None) == 1   # blend_masks NULL
    assert F(0x1000, 5, 0x1000, 0x1000, 10, 16, 16, None, 4, 0x1000, 0x1000, 0x1000, None, 0x1000,
             None, None, None, None, None) == 1   # stats outputs NULL
    assert F(0x1000, 5, 0x1000, 0x1000, 10, 16, 16, None, 8, 0x1000, 0x1000, 0x1000, None, 0x1000,
             None, None, 0x1000, None, None) == 1   # distortion totals NULL
    assert F(0x1000, 5, 0x1000, 0x1000, 10, 16, 16, None, 8, 0x1000, 0x1000, 0x1000, None, 0x1000,
             None, None, 0x1000, 0x1008, None) == 1   # totals not 16-byte aligned
    assert "aligned" in lib.ss_last_error().decode()
    # backward: NULL gradient array, accum flag without buffer or workspace, distortion inputs
    B = lambda flags, g, ws=None, nbytes=0, acc=None, dt=None, dd=None, rec=0x1000, masks=0x1000: \
        lib.ss_raster_bwd_records(rec, 4, 0x1000, 0x1000, 8, 16, 16, None, flags, 0x1000, 0x1000,
                                  masks, 0x1000, dt, dd, ctypes.byref(g), acc, ws, nbytes,
                                  None)  # noqa: E731
    g = SsGrads(0x1000, None, 0x1000, 0x1000, None)
    assert B(0, g) == 1
    g = SsGrads(0x1000, 0x1000, 0x1000, 0x1000, None)
    assert B(1, g, ws=0x1000, nbytes=1 << 20) == 1            # accum without buffer
    assert B(1, g, ws=0x1000, nbytes=8, acc=0x1000) == 1      # small workspace
    assert B(0, g, rec=None) == 1
    assert B(0, g, masks=None) == 1                          # masks rebuilt: needs a workspace
    assert B(0, g, masks=None, ws=0x1000, nbytes=1000) == 1
    assert "blend masks" in lib.ss_last_error().decode()
    assert B(32, g, ws=0x1000, nbytes=1 << 20) == 1           # unknown flag
    # SS_RECORDS_CLEARED is the backward's: the forward rejects it (the
    # static-scratch backward accepts and ignores it); unknown bits are rejected
    assert F(0x1000, 5, 0x1000, 0x1000, 10, 16, 16, None, 16, 0x1000, 0x1000, 0x1000, None,
             0x1000, None, None, None, None, None) == 1
    assert lib.ss_raster_bwd_noalloc(0x1000, 4, 0x1000, 0x1000, 8, 16, 16, None, 32, 0x1000,
                                     0x1000, 0x1000, 0x1000, ctypes.byref(g), None, None) == 1
    # the forward's optional bwd_workspace: 256-byte aligned and large enough for the records
    Fw = lambda ws, nbytes: lib.ss_raster_fwd_records(  # noqa: E731
        0x1000, 5, 0x1000, 0x1000, 10, 16, 16, None, 0, 0x1000, 0x1000, 0x1000, None, 0x1000, None,
        None, None, None, ws, nbytes, None)
    assert Fw(0x1010, 1 << 20) == 1
    assert "aligned" in lib.ss_last_error().decode()
    assert Fw(0x1000, 8) == 1
    assert "bwd_workspace" in lib.ss_last_error().decode()
    assert B(8, g, ws=0x1000, nbytes=1 << 20, dt=0x1000) == 1   # dL_ddist NULL
    assert B(8, g, ws=0x1000, nbytes=1 << 20, dt=0x1008, dd=0x1000) == 1   # misaligned totals
    assert B(8, g, ws=0x1000, nbytes=1 << 20, dt=0x1000, dd=0x1000) == 1   # ddepth NULL
    assert "ddepth" in lib.ss_last_error().decode()
    assert lib.ss_raster_bwd_noalloc(0x1000, 4, 0x1000, 0x1000, 8, 16, 16, None, 8, 0x1000,
                                     0x1000, 0x1000, 0x1000, ctypes.byref(g), None, None) == 5
    # the entry points that take the splats themselves
    S = ctypes.byref(sp)
    Fs = lambda flags, img=0x1000, spl=S: lib.ss_raster_fwd(  # noqa: E731
        spl, 0x1000, 0x1000, 16, 16, None, flags, img, 0x1000, 0x1000, None, None)
    assert Fs(0, spl=None) == 1
    assert Fs(0, img=None) == 1
    assert Fs(2) == 1                                        # median without its buffer
    assert Fs(4) == 5 and Fs(8) == 5                         # statistics, distortion
    assert "ss_raster_fwd_records" in lib.ss_last_error().decode()
    assert Fs(64) == 1                                       # unknown flag
    Bs = lambda flags, ws=0x1000, nbytes=1 << 20, spl=S, acc=0x1000: lib.ss_raster_bwd(  # noqa: E731
        spl, 0x1000, 0x1000, 16, 16, None, flags, 0x1000, 0x1000, 0x1000, ctypes.byref(g), acc, ws,
        nbytes, None)
    assert Bs(0, spl=None) == 1
    assert Bs(8) == 5                                        # distortion
    assert Bs(16) == 1                                       # records-cleared flag
    assert Bs(1, acc=None) == 1                              # accum without buffer
    assert Bs(0, ws=0x1010) == 1                             # misaligned workspace
    assert Bs(0, nbytes=256) == 1                            # no room for records and masks
    assert "workspace" in lib.ss_last_error().decode()
    unaligned = SsSplats(0x1004, 0x1000, 0x1000, 0x1000, 0x1000, 4)
    assert Bs(0, spl=ctypes.byref(unaligned)) == 1
    # pair count / sort status with NULL
    assert lib.ss_pair_count(None, 0, None, None, None) == 1
    assert lib.ss_sort_status(None, None) == 1
    assert lib.ss_probe_red_f32(None, 1, 1, None) == 1


def test_missing_library_fails_loudly(tmp_path):
    from gaussian_splatting_differentiable_gb300 import _lib
    with pytest.raises(ImportError):
        _lib.load(str(tmp_path / "nope.so"))


def test_projection_rejects_bad_arguments_on_the_host(lib):
    from gaussian_splatting_differentiable_gb300._lib import SsCamera, SsGrads3d, SsSplats3d

    def cam(**kw):
        c = SsCamera()
        for k in range(9):
            c.R[k] = 1.0 if k in (0, 4, 8) else 0.0
        c.fx = c.fy = 100.0
        c.cx, c.cy, c.near_z, c.blur = 32.0, 32.0, 0.2, 0.3
        for k, v in kw.items():
            setattr(c, k, v)
        return c
    s = SsSplats3d(0x1000, 0x1000, 0x1000, 0x1000, 10, 3)
    g = SsGrads3d(0x1000, 0x1000, 0x1000, 0x1000)
    P = ctypes.byref
    assert lib.ss_project_fwd(None, P(cam()), 0x1000, 0x1000, 0x1000, 0x1000, None) == 1
    assert lib.ss_project_fwd(P(s), None, 0x1000, 0x1000, 0x1000, 0x1000, None) == 1
    bad_deg = SsSplats3d(0x1000, 0x1000, 0x1000, 0x1000, 10, 4)
    assert lib.ss_project_fwd(P(bad_deg), P(cam()), 0x1000, 0x1000, 0x1000, 0x1000, None) == 1
    assert "sh_degree" in lib.ss_last_error().decode()
    misaligned = SsSplats3d(0x1000, 0x1000, 0x1004, 0x1000, 10, 3)
    assert lib.ss_project_fwd(P(misaligned), P(cam()), 0x1000, 0x1000, 0x1000, 0x1000, None) == 1
    null_sh = SsSplats3d(0x1000, 0x1000, 0x1000, None, 10, 3)
    assert lib.ss_project_fwd(P(null_sh), P(cam()), 0x1000, 0x1000, 0x1000, 0x1000, None) == 1
    assert lib.ss_project_fwd(P(s), P(cam(fx=0.0)), 0x1000, 0x1000, 0x1000, 0x1000, None) == 1
    assert lib.ss_project_fwd(P(s), P(cam(blur=float("nan"))), 0x1000, 0x1000, 0x1000, 0x1000,
                              None) == 1
    assert lib.ss_project_fwd(P(s), P(cam()), 0x1004, 0x1000, 0x1000, 0x1000, None) == 1
    assert lib.ss_project_fwd(P(s), P(cam()), None, 0x1000, 0x1000, 0x1000, None) == 1
    assert lib.ss_project_bwd(P(s), P(cam()), 0x1000, None, 0x1000, P(g), None) == 1
    assert lib.ss_project_bwd(P(s), P(cam()), 0x1000, 0x1000, 0x1000, None, None) == 1
    g_mis = SsGrads3d(0x1000, 0x1000, 0x1008, 0x1000)
    assert lib.ss_project_bwd(P(s), P(cam()), 0x1000, 0x1000, 0x1000, P(g_mis), None) == 1
    empty = SsSplats3d(None, None, None, None, 0, 3)
    assert lib.ss_project_fwd(P(empty), P(cam()), None, None, None, None, None) == 0
    assert lib.ss_project_bwd(P(empty), P(cam()), None, None, None, P(g), None) == 0


def test_ssim_rejects_bad_arguments_on_the_host(lib):
    assert lib.ss_ssim_workspace_bytes(3, 822, 1237) == 16 * 3 * 26 * 39 + 16
    assert lib.ss_ssim_workspace_bytes(0, 8, 8) == 0
    ws = 16 * 3 + 16
    assert lib.ss_ssim_loss(0x1000, 0x1000, 0, 8, 8, 0.2, 0x1000, 0x1000, 0x1000, ws, None) == 5
    assert lib.ss_ssim_loss(0x1000, 0x1000, 3, 8, 40000, 0.2, 0x1000, 0x1000, 0x1000, ws, None) == 5
    assert lib.ss_ssim_loss(None, 0x1000, 3, 8, 8, 0.2, 0x1000, 0x1000, 0x1000, ws, None) == 1
    assert lib.ss_ssim_loss(0x1000, 0x1000, 3, 8, 8, 1.5, 0x1000, 0x1000, 0x1000, ws, None) == 1
    assert lib.ss_ssim_loss(0x1000, 0x1000, 3, 8, 8, float("nan"), 0x1000, 0x1000, 0x1000, ws,
                            None) == 1
    assert lib.ss_ssim_loss(0x1000, 0x1000, 3, 8, 8, 0.2, 0x1000, 0x1000, 0x1008, ws, None) == 1
    assert lib.ss_ssim_loss(0x1000, 0x1000, 3, 8, 8, 0.2, 0x1000, 0x1000, 0x1000, ws - 1, None) == 1
    assert "workspace" in lib.ss_last_error().decode()


def test_binding_rejects_a_short_counters_buffer():
    """The counters cross the C ABI as a plain pointer; the binding checks that
    the tensor holds the four 64-bit words the library writes."""
    torch = pytest.importorskip("torch")
    import gaussian_splatting_differentiable_gb300 as ss
    short = torch.zeros(2, dtype=torch.int64)
    with pytest.raises(ValueError, match="four|4 64-bit"):
        ss.ss_pair_count(short, 10)
    keys = torch.zeros(4, dtype=torch.int64)
    vals = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(ValueError):
        ss.ss_sort_pairs_dev(keys, vals, short, 4, 16, 16, torch.zeros(2, dtype=torch.int32),
                             torch.zeros(256, dtype=torch.uint8), stream=0)
