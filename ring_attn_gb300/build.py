"""Builds libringattn.so in-tree for sm_103a (nvcc, one translation unit per kernel family, in parallel).

build(debug_bounds=True) builds the debug variant libringattn_dbg.so instead:
the same sources compiled with RA_DEBUG_BOUNDS, under which every kernel checks
its tiled-copy coordinates and global row indices against the tensor extents
and reports a violation as RA_ERR_DEVICE (with the site) instead of making the
access.  The binding loads it when RA_LIB_VARIANT=debug_bounds is set."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libringattn.so")
BUILD_DBG = os.path.join(PKG, "_build_dbg")
LIB_DBG = os.path.join(PKG, "libringattn_dbg.so")
SOURCES = ["ra_api.cu", "ra_fwd.cu", "ra_bwd.cu", "ra_dkdv_pair.cu", "ra_simple.cu"]
HEADERS = [os.path.join(CSRC, h) for h in ("ra_device.cuh", "ra_internal.h", "ra_tiles.cuh", "ra_bwd_common.cuh")] + [
    os.path.join(ROOT, "include", "ringattn.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libringattn.so")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build(verbose: bool = False, force: bool = False, debug_bounds: bool = False) -> str:
    """Compile every CUDA source for sm_103a and link libringattn.so (or, with
    debug_bounds, libringattn_dbg.so); returns its path."""
    nvcc = _nvcc()
    bdir, lib = (BUILD_DBG, LIB_DBG) if debug_bounds else (BUILD, LIB)
    extra = ["-DRA_DEBUG_BOUNDS"] if debug_bounds else []
    os.makedirs(bdir, exist_ok=True)
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(bdir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + HEADERS):
            cmd = [nvcc] + ARCH + FLAGS + extra + (["-Xptxas", "-v"] if verbose else []) + ["-c", s, "-o", o]
            jobs.append(cmd)
    if jobs:
        with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for out in ex.map(_run, jobs):
                if verbose and out:
                    sys.stdout.write(out)
    if force or jobs or _stale(lib, objs):
        _run([nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", lib] + objs)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, debug_bounds="--debug-bounds" in sys.argv))
