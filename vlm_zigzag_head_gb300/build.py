"""Builds libcpattn.so (sm_103a) in-tree with nvcc; no cmake, no torch build.

Objects go to ``_build/`` at the repository root, the library to
``vlm_zigzag_head_gb300/_lib/libcpattn.so``.  Translation units compile in
parallel and are skipped when newer than every source and header.

``build(checked=True)`` makes the bounds-checked debug library instead
(``-DCPATTN_BOUNDS_CHECK``; objects in ``_build_checked/``, library
``_lib/libcpattn_checked.so``): its kernels test every row and head index
before a TMA load, TMA reduce or global store and report a failure through
the workspace status word (CP_ERR_BOUNDS) instead of touching the address.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libcpattn.so")
BUILD_CHECKED = os.path.join(ROOT, "_build_checked")
LIB_CHECKED = os.path.join(LIBDIR, "libcpattn_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _headers():
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))


def _compile(src, extra, verbose, build_dir=BUILD, defines=()):
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    newest = max([os.path.getmtime(src)] + [os.path.getmtime(h) for h in _headers()])
    if os.path.exists(obj) and os.path.getmtime(obj) >= newest and not extra:
        return obj, ""
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + list(defines) + list(extra) + ["-c", src, "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
    return obj, r.stdout + r.stderr


def build(verbose: bool = False, extra=(), jobs: int = 0, checked: bool = False) -> str:
    build_dir, lib = (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)
    defines = ["-DCPATTN_BOUNDS_CHECK"] if checked else []
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    srcs = sources()
    jobs = jobs or min(len(srcs), os.cpu_count() or 4)
    with ThreadPoolExecutor(max_workers=jobs) as ex:
        results = list(ex.map(lambda s: _compile(s, extra, verbose, build_dir, defines), srcs))
    objs = [o for o, _ in results]
    for _, log in results:
        if log.strip() and verbose:
            print(log)
    newest = max(os.path.getmtime(o) for o in objs)
    if not os.path.exists(lib) or os.path.getmtime(lib) < newest or extra:
        cmd = [nvcc()] + ARCH + ["-shared", "-o", lib] + objs + ["-lpthread"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    return lib


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas" in sys.argv else []
    print(build(verbose=v or bool(extra), extra=extra, checked="--checked" in sys.argv))
