"""Build libsgemm_gb300.so in-tree with nvcc for sm_103a.

Each csrc/*.cu file compiles to an object in parallel (one -gencode, no
fast-math, -lineinfo for profiling), then nvcc links them into a shared
library next to this file.  ptxas register/spill reports go to
_build/ptxas_<unit>.log.  Rebuilds only when a source or header is newer
than the library (or force=True).  Runs without a GPU.

build(checked=True) makes the checked build, libsgemm_gb300_checked.so
(objects in _build_checked/): the same sources compiled with
-DSGEMM_CHECKED, whose kernels test every hand-computed shared-memory and
workspace index before the access (csrc/checked.cuh).  Tests load it with
SGEMM_GB300_LIBRARY=checked.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libsgemm_gb300.so")
# the checked build: the same sources with -DSGEMM_CHECKED (csrc/checked.cuh)
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libsgemm_gb300_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-Wformat,-Werror=format", "-Xptxas", "-v",
              "--expt-relaxed-constexpr", "-I", CSRC, "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsgemm_gb300.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date(checked: bool = False) -> bool:
    lib = LIB_CHECKED if checked else LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _compile(src: str, checked: bool = False) -> str:
    unit = os.path.splitext(os.path.basename(src))[0]
    out_dir = BUILD_CHECKED if checked else BUILD
    obj = os.path.join(out_dir, unit + ".o")
    cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, *(["-DSGEMM_CHECKED"] if checked else []), "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(out_dir, f"ptxas_{unit}.log"), "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {unit}.cu:\n{r.stderr[-6000:]}")
    return obj


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Build the library (checked=True: the checked build, libsgemm_gb300_checked.so)."""
    lib = LIB_CHECKED if checked else LIB
    out_dir = BUILD_CHECKED if checked else BUILD
    if not force and up_to_date(checked):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    srcs = _sources()
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda src: _compile(src, checked), srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, lib)
    if verbose:
        for log in sorted(glob.glob(os.path.join(out_dir, "ptxas_*.log"))):
            with open(log) as f:
                sys.stdout.write(f.read())
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))
