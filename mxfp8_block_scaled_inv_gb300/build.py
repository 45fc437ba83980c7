"""Build libmxq.so in-tree for sm_103a.

Each CUDA translation unit is compiled by nvcc in parallel with
``-gencode arch=compute_103a,code=sm_103a``, the C-ABI layer by the host
compiler, and the objects are linked into ``libmxq.so`` next to this file.
A build is skipped when the library is newer than every source and header.
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
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libmxq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CU_SOURCES = ["quant.cu", "misc.cu", "bmm.cu", "linear_noalloc.cu", "kv_insert.cu"]
CXX_SOURCES = ["api.cpp"]


def cuda_home() -> str:
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return cand
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    raise RuntimeError("nvcc not found (set CUDA_HOME)")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "mxq.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}")
    return r.stdout


def build(verbose: bool = False, force: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link libmxq.so; returns its path."""
    if not force and up_to_date():
        return LIB_PATH
    home = cuda_home()
    nvcc = os.path.join(home, "bin", "nvcc")
    os.makedirs(BUILD_DIR, exist_ok=True)
    inc = ["-I", INCLUDE, "-I", CSRC, "-I", os.path.join(home, "include")]
    jobs = []
    for src in CU_SOURCES:
        obj = os.path.join(BUILD_DIR, src + ".o")
        cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
               "--expt-relaxed-constexpr", *inc, "-c", os.path.join(CSRC, src), "-o", obj]
        if ptxas_info:
            cmd.insert(1, "-Xptxas=-v")
        jobs.append((cmd, obj))
    cxx = os.environ.get("CXX", "g++")
    for src in CXX_SOURCES:
        obj = os.path.join(BUILD_DIR, src + ".o")
        cmd = [cxx, "-O2", "-std=c++17", "-fPIC", "-Wall", *inc, "-c", os.path.join(CSRC, src),
               "-o", obj]
        jobs.append((cmd, obj))
    outputs = []
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        for out in ex.map(lambda j: _run(j[0], verbose), jobs):
            outputs.append(out)
    if ptxas_info:
        print("\n".join(outputs))
    tmp = LIB_PATH + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *[o for _, o in jobs],
          "-L", os.path.join(home, "lib64")], verbose)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(verbose=True, force="--force" in sys.argv, ptxas_info="--ptxas-info" in sys.argv)
    print(LIB_PATH)
