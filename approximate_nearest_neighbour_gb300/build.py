"""Builds libivfpq_gb300.so from csrc/ with nvcc for sm_103a (in-tree).

Each .cu file is compiled to an object in parallel, then the objects are
linked into a shared library next to this file. The CUDA runtime is linked
statically, so loading the library needs no GPU driver (only calling into it
does).
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libivfpq_gb300.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)
# the debug build: device bounds checks (-DIVFPQ_DEBUG_CHECKS) that record a
# failure in the device status word instead of trapping
DEBUG_BUILD_DIR = os.path.join(HERE, "_build_debug")
DEBUG_LIB_PATH = os.path.join(HERE, "libivfpq_gb300_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return (glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build_library(force: bool = False, verbose: bool = False, jobs: int | None = None,
                  debug: bool = False) -> str:
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    flags = NVCC_FLAGS + (["-DIVFPQ_DEBUG_CHECKS"] if debug else [])
    os.makedirs(build_dir, exist_ok=True)
    srcs = _sources()
    hdrs = _headers()
    objs = []
    todo = []
    for src in srcs:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + hdrs):
            todo.append((src, obj))
    exe = nvcc()

    def compile_one(item):
        src, obj = item
        cmd = [exe] + ARCH + flags + ["-c", src, "-o", obj + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr[-4000:]}")
        os.replace(obj + ".tmp", obj)
        if verbose:
            print("compiled", os.path.basename(src), flush=True)

    if todo:
        n = jobs or max(1, min(len(todo), os.cpu_count() or 1))
        with cf.ThreadPoolExecutor(n) as ex:
            list(ex.map(compile_one, todo))
    if force or todo or _stale(lib_path, objs):
        tmp = lib_path + f".{os.getpid()}.tmp"
        cmd = [exe] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build_library(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))
