"""Build step for the CUDA library: compiles csrc/ for sm_103a and links
libfp8lin.so in-tree (next to this file).  Translation units are compiled in
parallel; nothing is installed anywhere.

    python -m fp8_mixed_precision_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfp8lin.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I" + INCLUDE] + ARCH
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall", "-I" + INCLUDE]

CU_SOURCES = ["quantize.cu", "gemm.cu", "glue.cu", "noalloc.cu"]
CXX_SOURCES = ["api.cpp"]


def _cuda_home() -> str:
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.exists(os.path.join(c, "bin", "nvcc")):
            return c
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    raise RuntimeError("nvcc not found")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + \
            [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)] + [os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


def _run(cmd, verbose, log=None):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if log:
        with open(log, "w") as f:
            f.write(r.stdout + r.stderr)
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)
    return r


def build(force: bool = False, verbose: bool = False, extra_nvcc=()) -> str:
    """Compile and link the library if any source is newer than it; return its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime():
        return LIB
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    os.makedirs(BUILD, exist_ok=True)
    jobs = []
    for f in CU_SOURCES:   # ptxas resource report (registers, spills) kept beside the object
        obj = os.path.join(BUILD, f + ".o")
        jobs.append(([nvcc, *NVCC_FLAGS, "-Xptxas", "-v", *extra_nvcc, "-c", os.path.join(CSRC, f),
                      "-o", obj], os.path.join(BUILD, f + ".ptxas.txt")))
    for f in CXX_SOURCES:
        obj = os.path.join(BUILD, f + ".o")
        jobs.append((["g++", *CXX_FLAGS, "-I" + os.path.join(cuda, "include"), "-c",
                      os.path.join(CSRC, f), "-o", obj], None))
    with ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
        list(ex.map(lambda c: _run(c[0], verbose, c[1]), jobs))
    objs = [os.path.join(BUILD, f + ".o") for f in CU_SOURCES + CXX_SOURCES]
    tmp = LIB + ".tmp"
    _run([nvcc, "-shared", *ARCH, "-o", tmp, *objs], verbose)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose))
    sys.exit(0)
