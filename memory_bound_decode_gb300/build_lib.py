"""Build libgemv.so in-tree for sm_103a.

Each translation unit compiles in its own nvcc process (in parallel), then one
nvcc call links the shared library. The result lands in
memory_bound_decode_gb300/_lib/libgemv.so (git-ignored). The CUDA runtime is
linked dynamically, with an rpath to the toolkit, so the library shares the
runtime that PyTorch loads.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_lib")
OBJ_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libgemv.so")

SOURCES = [
    "gemv_fma_instances.cu",
    "gemv_fma_instances_b3_8.cu",
    "gemv_fma_instances_b9_16.cu",
    "gemv_mma_instances_nb1.cu",
    "gemv_mma_instances_nb2.cu",
    "gemv_w4_instances.cu",
    "gemv_fp8_instances.cu",
    "gemv_tc_instances.cu",
    "gemv_streamk_instances.cu",
    "gemv_noalloc.cu",
    "gemv_dispatch.cu",
    "planner.cpp",
    "gemv_api.cpp",
]
HEADERS = ["gemv_internal.h", "gemv_common.cuh", "gemv_kernel.cuh", "gemv_mma_kernel.cuh", "gemv_w4_kernel.cuh",
           "gemv_tc_kernel.cuh",
           "gemv_streamk_kernel.cuh", "gemv_fp8_kernel.cuh", os.path.join("..", "..", "include", "gemv.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home:
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def nvcc() -> str:
    return os.path.join(cuda_home(), "bin", "nvcc")


def _flags(extra=()) -> list[str]:
    return ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", *ARCH, *extra]


def _newest(paths) -> float:
    return max(os.path.getmtime(p) for p in paths)


LIB_DEBUG = os.path.join(OUT_DIR, "libgemv_debug.so")
DEBUG_FLAGS = ("-DGEMV_DEBUG_WRITECOUNT",)
LIB_DEBUG_DROP_X = os.path.join(OUT_DIR, "libgemv_debug_drop_x.so")
DROP_X_FLAGS = ("-DGEMV_DEBUG_DROP_X",)


def build_debug(force: bool = False, verbose: bool = False) -> str:
    """The test build that counts output stores (gemv_debug_write_count)."""
    return build(force=force, verbose=verbose, extra_flags=DEBUG_FLAGS, lib=LIB_DEBUG)


def build_debug_drop_x(force: bool = False, verbose: bool = False) -> str:
    """The test build whose tcgen05 kernels never issue their copies of x: the
    stages' barriers wait for bytes that never come, so the bounded waits run
    out (limit 2^14 rounds in this build) and the kernel takes its failure
    path: NaN outputs, the status bit, its tensor memory freed."""
    return build(force=force, verbose=verbose, extra_flags=DROP_X_FLAGS, lib=LIB_DEBUG_DROP_X)


def build(force: bool = False, verbose: bool = False, extra_flags=(), lib: str = LIB) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    os.makedirs(OBJ_DIR, exist_ok=True)
    headers = [os.path.normpath(os.path.join(CSRC, h)) for h in HEADERS]
    tag = "" if not extra_flags else "_" + hashlib.sha256("\0".join(extra_flags).encode()).hexdigest()[:10]
    hdr_time = _newest(headers)

    def compile_one(src: str) -> str:
        path = os.path.join(CSRC, src)
        obj = os.path.join(OBJ_DIR, os.path.splitext(src)[0] + tag + ".o")
        if (not force and os.path.exists(obj)
                and os.path.getmtime(obj) >= max(os.path.getmtime(path), hdr_time)):
            return obj
        cmd = [nvcc(), *_flags(extra_flags), "-c", path, "-o", obj]
        if src.endswith(".cpp"):
            cmd[1:1] = ["-x", "cu"]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.run(cmd, check=True)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))

    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest(objs):
        return lib
    tmp = f"{lib}.{os.getpid()}.tmp"
    libdir = os.path.join(cuda_home(), "lib64")
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", f"-rpath,{libdir}"]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
