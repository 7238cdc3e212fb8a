"""Build libdpz.so in-tree with nvcc for sm_103a (no cmake, one -gencode).

Translation units compile in parallel; the shared library links the CUDA
runtime statically, so loading it needs no GPU.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdpz.so")

SOURCES = ["api.cpp", "reduce.cu", "adamw.cu", "staged.cu", "norm_static.cu"]
HEADERS = [os.path.join(CSRC, h) for h in ("internal.h", "device.cuh", "bulk.cuh")] + \
    [os.path.join(INCLUDE, "dpz.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    # IEEE division and square root, no flush-to-zero, no contraction into FMA:
    # the arithmetic is bit-for-bit the documented operation sequence
    "-prec-div=true", "-prec-sqrt=true", "-ftz=false", "-fmad=false",
    "-Xcompiler", "-fPIC,-fvisibility=hidden,-ffp-contract=off",
    "-I" + INCLUDE, "-I" + CSRC,
]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str) -> str:
    path = os.path.join(CSRC, src)
    obj = os.path.join(BUILD, src + ".o")
    if _stale(obj, [path] + HEADERS):
        subprocess.check_call([_nvcc(), *NVCC_FLAGS, "-c", path, "-o", obj])
    return obj


def build(verbose: bool = False) -> str:
    """Compile (if anything changed) and return the path of libdpz.so."""
    os.makedirs(BUILD, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(_compile, SOURCES))
    if _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call([_nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared",
                               "-Xcompiler", "-fPIC", *objs, "-o", tmp])
        os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}", file=sys.stderr)
    return LIB


if __name__ == "__main__":
    build(verbose=True)
