"""Build the C-ABI library ``_build/libsa_gb300.so`` for sm_103a.

Each translation unit is compiled in parallel with nvcc (device code for
compute_103a/sm_103a only) and linked into one shared object with the CUDA
runtime linked statically, so the library loads without a GPU driver (the
symbol-export test runs on machines without one).

``build(debug=True)`` makes the SA_DEBUG variant ``_build_debug/libsa_gb300_debug.so``:
the same kernels with device-side range checks of every work description
(a failed check sets the error word and the item is skipped), plus the
test entry point declared in ``include/sa_debug.h``.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIBNAME = "libsa_gb300.so"
LIBPATH = os.path.join(BUILD, LIBNAME)
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIBPATH_DEBUG = os.path.join(BUILD_DEBUG, "libsa_gb300_debug.so")

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-std=c++17", "-O3", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, headers, extra, build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    if not _stale(obj, [src] + headers + [__file__]):
        return obj
    cmd = [NVCC] + COMMON + extra + ["-c", src, "-o", obj]
    if src.endswith(".cu"):
        cmd[1:1] = ARCH + ["-lineinfo", "-Xptxas", "-v"] if os.environ.get("SA_PTXAS_V") else ARCH + ["-lineinfo"]
    else:
        cmd = [NVCC] + COMMON + extra + ["-x", "c++", "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, extra=(), debug: bool = False) -> str:
    """Compile and link; returns the library path.  Rebuilds what is stale."""
    build_dir = BUILD_DEBUG if debug else BUILD
    libpath = LIBPATH_DEBUG if debug else LIBPATH
    extra = list(extra) + (["-DSA_DEBUG=1"] if debug else [])
    os.makedirs(build_dir, exist_ok=True)
    srcs = sources()
    headers = sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")))
    if force:
        for o in glob.glob(os.path.join(build_dir, "*.o")):
            os.remove(o)
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, headers, extra, build_dir), srcs))
    if force or _stale(libpath, objs):
        tmp = libpath + ".tmp"
        cmd = [NVCC] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, libpath)
    return libpath


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, debug="--debug" in sys.argv))
