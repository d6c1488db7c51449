"""Build libhfa.so (the CUDA library) in-tree with nvcc for sm_103a.

Each .cu file compiles to an object in parallel, then nvcc links the shared library
against the shared CUDA runtime.  Nothing here needs a GPU: nvcc cross-compiles.
Usage: python -m quantized_attention_layer_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libhfa.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libhfa")


def cuda_home() -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc())))


def _flags(verbose: bool):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                "--expt-relaxed-constexpr", "-Xcompiler", "-Wall,-Wno-unused-function"]
    if verbose:
        f += ["-Xptxas", "-v"]
    return f


def _headers():
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def build(force: bool = False, verbose: bool = False) -> str:
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    os.makedirs(BUILD, exist_ok=True)
    newest_header = max((os.path.getmtime(h) for h in _headers()), default=0)
    jobs = []
    for src in srcs:
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        stale = force or not os.path.exists(obj) or \
            os.path.getmtime(obj) < max(os.path.getmtime(src), newest_header)
        jobs.append((src, obj, stale))
    cmd0 = [nvcc()] + _flags(verbose)

    def compile_one(job):
        src, obj, stale = job
        if not stale:
            return obj, ""
        p = subprocess.run(cmd0 + ["-c", src, "-o", obj], capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{p.stdout}\n{p.stderr}")
        return obj, p.stderr

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(compile_one, jobs))
    if verbose:
        for obj, log in results:
            if log:
                print(f"== {os.path.basename(obj)}\n{log}", file=sys.stderr)
    objs = [o for o, _ in results]
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        libdir = os.path.join(cuda_home(), "lib64")
        tmp = LIB + f".tmp{os.getpid()}"
        link = [nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs + \
            ["-Xlinker", f"-rpath,{libdir}"]
        p = subprocess.run(link, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"link failed:\n{p.stdout}\n{p.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
