"""Compile the CUDA sources of this package into libfa.so (sm_103a), in place.

Each translation unit is compiled by its own nvcc process (in parallel), then
the objects are linked into ``libfa.so`` next to this file.  The CUDA runtime
is linked statically, and the driver's tensor-map encoder is looked up at run
time, so the library loads on a machine without a GPU driver (for the
symbol-export tests) and runs on any sm_103 device.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfa.so")
# the debug build: kernels with index checks (FA_DEBUG), objects and library of its own
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libfa_debug.so")
SOURCES = ["fa_api.cu", "fwd_tc.cu", "fwd_f32.cu", "bwd_tc.cu", "bwd_aux.cu", "fa_noalloc.cu", "fwd_fp8.cu"]
HEADERS = ["ptx.cuh", "internal.h", "bwd_sched.cuh", "fp8.h", "tiles.cuh", "fwd_common.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa.so")


def _deps():
    return ([os.path.join(CSRC, s) for s in SOURCES] + [os.path.join(CSRC, h) for h in HEADERS]
            + [os.path.join(ROOT, "include", "fa.h"), os.path.abspath(__file__)])


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _compile(src: str, extra: list[str], build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-I", os.path.join(ROOT, "include"), *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if "-v" in extra and r.stderr:
        print(r.stderr, end="")
    return obj


def build(force: bool = False, extra_flags: list[str] | None = None, verbose: bool = False,
          debug: bool = False) -> str:
    """Build libfa.so (debug: libfa_debug.so, with the kernels' index checks) if any
    source is newer than it (or if forced); returns its path."""
    lib, build_dir = (LIB_DEBUG, BUILD_DEBUG) if debug else (LIB, BUILD)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    extra = list(extra_flags or [])
    if debug:
        extra += ["-DFA_DEBUG"]
    if verbose:
        extra += ["-Xptxas", "-v"]
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, build_dir), SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
