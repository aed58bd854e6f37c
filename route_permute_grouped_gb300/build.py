"""Build the CUDA library in-tree: every .cu file under csrc/ compiled for
sm_103a in parallel, linked into ``_lib/libmoe_gb300.so`` (static CUDA runtime,
no link-time libcuda, so the library loads on a machine without a GPU).

``build(checked=True)`` builds the bounds-check variant instead
(``_lib/libmoe_gb300_checked.so``, compiled with ``-DMOE_BOUNDS_CHECK``: the
element-wise kernels range-check every row and expert index they read and
record MOE_ERR_DEVICE_INDEX instead of reading out of range). The binding loads
it when the environment sets ``MOE_BOUNDS_CHECK=1``.

Usage: ``python -m route_permute_grouped_gb300.build [--checked]`` (or
``build()``). Rebuilds only when a source or header is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_lib")
OBJ_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(OUT_DIR, "libmoe_gb300.so")
LIB_CHECKED = os.path.join(OUT_DIR, "libmoe_gb300_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-v"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h")) + [os.path.abspath(__file__)]


def up_to_date(checked: bool = False) -> bool:
    lib = LIB_CHECKED if checked else LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src: str, log: bool, checked: bool = False):
    obj_dir = OBJ_DIR + ("_checked" if checked else "")
    obj = os.path.join(obj_dir, os.path.basename(src).replace(".cu", ".o"))
    extra = ["-DMOE_BOUNDS_CHECK"] if checked else []
    cmd = [_nvcc(), *ARCH, *FLAGS, *extra, "-I", os.path.join(ROOT, "include"), "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
    if log:
        with open(obj + ".ptxas.txt", "w") as f:
            f.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile and link the library (the bounds-check variant with
    checked=True); returns its path."""
    lib = LIB_CHECKED if checked else LIB
    if not force and up_to_date(checked):
        return lib
    os.makedirs(OBJ_DIR + ("_checked" if checked else ""), exist_ok=True)
    os.makedirs(OUT_DIR, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda s: _compile(s, True, checked), srcs))
    tmp = lib + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        for o in objs:
            print(open(o + ".ptxas.txt").read())
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))
