"""Builds ``libpa.so`` (the C-ABI library) in-tree for sm_103a.

Each translation unit is compiled in parallel with nvcc (CUDA) or g++ (host
allocator) and linked with the static CUDA runtime, so the library loads on a
machine without a GPU driver and needs no driver library at link time.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libpa.so")

CUDA_SOURCES = ["pa_decode.cu", "pa_cache.cu", "pa_runtime.cu", "pa_noalloc.cu", "pa_multi_query.cu",
                "pa_multi_query_tc.cu", "pa_step.cu"]
CXX_SOURCES = ["pa_allocator.cpp"]
HEADERS = ["pa_common.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpa.so")


def _inputs():
    files = [os.path.join(CSRC, f) for f in CUDA_SOURCES + CXX_SOURCES + HEADERS]
    return files + [os.path.join(INCLUDE, "pa.h"), os.path.abspath(__file__)]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n%s\n%s" % (" ".join(cmd), r.stdout))
    return r.stdout


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compiles and links ``_build/libpa.so`` if any input is newer; returns its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC]
    jobs = []
    for f in CUDA_SOURCES:
        obj = os.path.join(BUILD, f + ".o")
        cmd = [nvcc, *ARCH, "-lineinfo", *common, "-Xcompiler", "-fPIC,-fvisibility=hidden",
               "-c", os.path.join(CSRC, f), "-o", obj]
        if ptxas_info:
            cmd.insert(1, "-Xptxas=-v")
        jobs.append((cmd, obj))
    for f in CXX_SOURCES:
        obj = os.path.join(BUILD, f + ".o")
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-fvisibility=hidden", "-I", INCLUDE, "-c",
               os.path.join(CSRC, f), "-o", obj]
        jobs.append((cmd, obj))
    logs = []
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        for out in ex.map(lambda j: _run(j[0]), jobs):
            logs.append(out)
    tmp = LIB + ".tmp%d" % os.getpid()
    _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[o for _, o in jobs]])
    os.replace(tmp, LIB)
    if verbose or ptxas_info:
        sys.stdout.write("".join(logs))
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
