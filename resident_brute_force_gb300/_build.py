"""Compile the CUDA library (librbf.so) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel to an object file under
``_build/`` and the objects are linked into ``librbf.so`` next to this file.
The CUDA runtime is linked statically, so the library loads without touching
the interpreter's own CUDA runtime.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "librbf.so")
# The checked variant (-DRBF_CHECKS: device-side bounds checks on the indices
# the kernels derive, reported through the error word).
CHECKS_BUILD_DIR = os.path.join(HERE, "_build_checks")
CHECKS_LIB_PATH = os.path.join(HERE, "librbf_checks.so")

SOURCES = ["engine.cu", "score_select.cu", "merge.cu", "topk_i32.cu", "noalloc.cu", "gemm_select.cu", "normalize.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librbf.so")


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "rbf.h"))
    return files


def is_stale(lib: str = LIB_PATH) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          checks: bool = False) -> str:
    """Build librbf.so (or, with ``checks``, librbf_checks.so) if any source is
    newer than it (or ``force``)."""
    lib = CHECKS_LIB_PATH if checks else LIB_PATH
    build_dir = CHECKS_BUILD_DIR if checks else BUILD_DIR
    if not force and not is_stale(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + list(extra_flags or []) + (["-DRBF_CHECKS"] if checks else [])

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib
