"""Build libpps.so in place: every CUDA translation unit for sm_103a, the host
planner with g++, linked with nvcc (static CUDA runtime, no libcuda link; the
driver API is reached through cudaGetDriverEntryPoint).

    python -m paged_prefix_shared_gb300.builder    # or build() from Python
"""
from __future__ import annotations

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
LIB = os.path.join(PKG, "libpps.so")

CUDA_SOURCES = ["api.cu", "kv_append.cu", "attn_bw.cu", "attn_mma.cu", "attn_tt.cu", "merge.cu", "noalloc.cu",
                "gemm.cu"]
CXX_SOURCES = ["planner.cpp", "radix_cache.cpp", "scheduler.cpp", "engine.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources_newer_than(target):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "pps.h"),
                                                                 __file__]
    return any(os.path.getmtime(f) > t for f in files if os.path.isfile(f))


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _sources_newer_than(LIB):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC]
    jobs = []
    for src in CUDA_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        jobs.append([nvcc, *ARCH, *common, "-lineinfo", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr", "-c", os.path.join(CSRC, src), "-o", obj])
    for src in CXX_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        jobs.append(["g++", *common, "-fPIC", "-Wall", "-c", os.path.join(CSRC, src), "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("build failed: " + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)

    with ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
        list(ex.map(run, jobs))
    objs = [os.path.join(BUILD, s + ".o") for s in CUDA_SOURCES + CXX_SOURCES]
    tmp = LIB + ".tmp"
    run([nvcc, *ARCH, "-shared", "-Xlinker", "--version-script=" + os.path.join(CSRC, "exports.map"),
         "-o", tmp, *objs])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
