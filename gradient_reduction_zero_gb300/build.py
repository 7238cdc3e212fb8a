"""Build libdpz.so in-tree with nvcc for sm_103a (no cmake, one -gencode),
then the CPython module _dpzcall that calls it from Python.

Translation units compile in parallel; the shared library links the CUDA
runtime statically, so loading it needs no GPU.  _dpzcall (csrc/pycall.c) is
plain C against Python.h and libdpz.so; where Python's headers are missing
the binding calls the library through ctypes instead.
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


PYCALL_SRC = os.path.join(CSRC, "pycall.c")


def pycall_path() -> str:
    import sysconfig
    return os.path.join(PKG, "_dpzcall" + sysconfig.get_config_var("EXT_SUFFIX"))


def build_pycall(verbose: bool = False) -> str | None:
    """Compile _dpzcall (if anything changed); None where Python's headers are
    not installed."""
    import sysconfig
    inc = sysconfig.get_paths()["include"]
    if not os.path.exists(os.path.join(inc, "Python.h")):
        if verbose:
            print(f"no Python.h under {inc}: the binding calls libdpz.so through ctypes",
                  file=sys.stderr)
        return None
    out = pycall_path()
    if _stale(out, [PYCALL_SRC, os.path.join(INCLUDE, "dpz.h"), LIB]):
        tmp = out + f".tmp{os.getpid()}"
        try:
            subprocess.check_call([os.environ.get("CC", "gcc"), "-O2", "-std=c11", "-shared",
                                   "-fPIC", "-I" + inc, "-I" + INCLUDE, PYCALL_SRC, "-L" + PKG,
                                   "-ldpz", "-Wl,-rpath,$ORIGIN", "-o", tmp])
        except (OSError, subprocess.CalledProcessError) as e:
            print(f"_dpzcall not built ({e}): the binding calls libdpz.so through ctypes",
                  file=sys.stderr)
            return None
        os.replace(tmp, out)
    if verbose:
        print(f"built {out}", file=sys.stderr)
    return out


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
    build_pycall(verbose)
    return LIB


if __name__ == "__main__":
    build(verbose=True)
