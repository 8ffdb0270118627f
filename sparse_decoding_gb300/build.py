"""Build the in-tree shared library ``libnmspmv.so`` for sm_103a with nvcc.

Each translation unit is compiled in parallel, then linked into one shared
library next to this file. No cmake, no torch extension machinery: the library
exposes a plain C ABI (``include/nmspmv.h``) and is loaded with ctypes.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libnmspmv.so")
# The bounds-checking variant (-DNM_BOUNDS_CHECK), built on request only.
BUILD_CHECK = os.path.join(HERE, "_build_check")
LIB_CHECK = os.path.join(HERE, "libnmspmv_check.so")

SOURCES = ["api.cu", "spmv.cu", "gemv.cu", "pack.cu", "noalloc.cu", "obs.cu", "tc_gemm.cu", "pack_host.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libnmspmv.so")


def _flags(src: str, check: bool = False):
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if check:
        common += ["-DNM_BOUNDS_CHECK"]
    if src.endswith(".cu"):
        return common + ARCH + ["-lineinfo", "-Xptxas", "-v", "--expt-relaxed-constexpr"]
    return common


def _compile(src: str, check: bool = False) -> tuple[str, str]:
    obj = os.path.join(BUILD_CHECK if check else BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj] + _flags(src, check)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "nmspmv.h"), __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, check: bool = False) -> str:
    """Compile and link; returns the library path. Rebuilds only when sources changed.

    check=True builds the bounds-checking variant libnmspmv_check.so instead
    (every data-dependent index checked; a violation is reported by
    nm_device_status as NM_ERR_BOUNDS and the access skipped)."""
    lib, bdir = (LIB_CHECK, BUILD_CHECK) if check else (LIB, BUILD)
    if not force and not _stale(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda src: _compile(src, check), SOURCES))
    with open(os.path.join(bdir, "ptxas.log"), "w") as f:
        for (obj, log), src in zip(results, SOURCES):
            f.write(f"==== {src}\n{log}\n")
    tmp = lib + f".tmp{os.getpid()}"
    cmd = ([nvcc(), "-shared", "-o", tmp] + [o for o, _ in results] + ARCH + ["-Xcompiler", "-fPIC"]
           + ["-ldl"])
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        print(open(os.path.join(bdir, "ptxas.log")).read())
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, check="--check" in sys.argv))
