"""Build libss.so (the C-ABI library) in-tree with nvcc for sm_103a.

    python gaussian_splatting_differentiable_gb300/build.py [-v] [--debug-bounds]

(run by path: importing the package loads the library this script builds)

Each .cu under csrc/ compiles to an object in parallel, then nvcc links them
into gaussian_splatting_differentiable_gb300/libss.so with the static CUDA
runtime, so the library needs nothing at run time beyond the driver.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build", "libss")
LIB = os.path.join(PKG, "libss.so")
# The variant with device-side bounds checks (-DSS_DEBUG_BOUNDS).
DEBUG_BUILD = os.path.join(ROOT, "_build", "libss_debug")
DEBUG_LIB = os.path.join(PKG, "libss_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def sources() -> list:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list:
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + \
        [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra: tuple = (),
          debug_bounds: bool = False) -> str:
    """Build libss.so, or with debug_bounds libss_debug.so (device-side
    bounds checks, SS_DEBUG_BOUNDS)."""
    lib, bdir = (DEBUG_LIB, DEBUG_BUILD) if debug_bounds else (LIB, BUILD)
    if debug_bounds:
        extra = tuple(extra) + ("-DSS_DEBUG_BOUNDS",)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ("-Xptxas", "-v") if v else ()
    print(build(force=True, verbose=v, extra=extra, debug_bounds="--debug-bounds" in sys.argv))
