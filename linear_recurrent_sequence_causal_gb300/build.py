"""Builds libprism.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` translation unit compiles in parallel to an object file;
the objects link into ``_build/libprism.so``.  Only sm_103a code is generated.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libprism.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libprism.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + [os.path.join(ROOT, "include", "prism.h"), os.path.abspath(__file__)])


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _deps())


DEBUG_LIB = os.path.join(BUILD, "debug", "libprism.so")


def build_debug(force: bool = False, jobs: int | None = None) -> str:
    """The bounds-checked debug build (-DPRISM_DEBUG_BOUNDS) in _build/debug/."""
    if not force and os.path.exists(DEBUG_LIB) and not any(
            os.path.getmtime(p) > os.path.getmtime(DEBUG_LIB) for p in _deps()):
        return DEBUG_LIB
    return _compile(DEBUG_LIB, os.path.join(BUILD, "debug", "obj"), ["-DPRISM_DEBUG_BOUNDS"], jobs)


def build(force: bool = False, jobs: int | None = None, verbose: bool = False) -> str:
    if not force and not stale():
        return LIB
    return _compile(LIB, os.path.join(BUILD, "obj"), [], jobs, verbose)


def _compile(lib: str, obj_dir: str, extra: list, jobs: int | None = None, verbose: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(obj_dir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    srcs = _sources()
    jobs = jobs or min(len(srcs), os.cpu_count() or 4)
    with concurrent.futures.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".{os.getpid()}.tmp"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
