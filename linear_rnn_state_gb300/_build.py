"""Builds the CUDA library (libwkv7.so) in-tree with nvcc for sm_103a.

The translation units compile in parallel, then link into one shared library
that uses the shared CUDA runtime (the same libcudart.so.13 PyTorch loads, so
both see the same current device).

It also links the debug build, libwkv7_debug.so: the same objects, the C ABI
and the WKV7 scan kernels recompiled with WKV7_DEBUG (every plain global load
and store checked against its buffer, 1 ms mbarrier wait limit, and the hooks
of include/wkv7_debug.h). Only the tests of those checks and of the timeout
path load it.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libwkv7.so")
DEBUG_LIB = os.path.join(PKG, "libwkv7_debug.so")
DEBUG_SOURCES = ["wkv7_api.cu", "wkv7_fwd2.cu", "wkv7_fwd3.cu", "wkv7_bwd2.cu", "wkv7_bwd3.cu",
                 "wkv7_bwd4.cu", "wkv7_bwd4_f32.cu"]  # recompiled with -DWKV7_DEBUG for the debug build

SOURCES = ["wkv7_api.cu", "wkv7_fwd2.cu", "wkv7_fwd3.cu", "wkv7_bwd2.cu", "wkv7_bwd3.cu", "wkv7_bwd4.cu",
           "wkv7_bwd4_f32.cu", "rwkv8_api.cu",
           "rwkv8_fwd.cu", "rwkv8_bwd.cu", "rwkv8_bwd_split.cu", "rwkv8_state.cu", "rwkv8_chunk.cu", "wkv7_epilogue.cu"]
HEADERS = ["wkv7_common.cuh", "wkv7_launch.h", "wkv7_mma.cuh", "wkv7_scaled.cuh", "wkv7_tmem.cuh", "wkv7_decay.cuh",
           "rwkv8_launch.h", "rwkv8_split.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-cudart", "shared",
                     "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the WKV7 CUDA library cannot be built")
    return path


def _cuda_lib_dir() -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc()))), "lib64")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile every .cu to an object (in parallel) and link libwkv7.so."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, h)
                                                          for h in ("wkv7.h", "rwkv8.h", "wkv7_debug.h")]
    objs, dobjs, jobs = [], [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + headers):
            jobs.append([nvcc(), *NVCC_FLAGS, *extra_flags, "-c", s, "-o", o])
        if src in DEBUG_SOURCES:
            o = os.path.join(BUILD_DIR, src.replace(".cu", ".debug.o"))
            if force or _stale(o, [s] + headers):
                jobs.append([nvcc(), *NVCC_FLAGS, *extra_flags, "-DWKV7_DEBUG", "-c", s, "-o", o])
        dobjs.append(o)

    def run(cmd):
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
        if verbose:
            print(res.stdout, res.stderr, sep="")

    with ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        list(ex.map(run, jobs))
    for lib, parts in ((LIB, objs), (DEBUG_LIB, dobjs)):
        if force or jobs or _stale(lib, parts):
            tmp = lib + f".tmp{os.getpid()}"
            run([nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *parts,
                 "-Xlinker", f"-rpath,{_cuda_lib_dir()}"])
            os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "-v" in sys.argv else []))
