"""Compile libfarn.so (the C ABI of include/farn.h) for sm_103a, in tree."""
from __future__ import annotations

import os
import subprocess
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libfarn.so")
SOURCES = [os.path.join(CSRC, "farn.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, "farn_kernels.cuh"),
                     os.path.join(INCLUDE, "farn.h")]
NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    # IEEE division and square root, denormals kept: the per-row rstd and
    # every bf16 rounding follow IEEE fp32 (no -use_fast_math, no -ftz).
    "-prec-div=true", "-prec-sqrt=true", "-ftz=false",
    "-Xcompiler", "-fPIC", "-shared",
]
_lock = threading.Lock()


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(p) > t for p in DEPENDS)


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Build libfarn.so next to this file if missing or older than its sources."""
    with _lock:
        if force or _stale():
            tmp = LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["nvcc", *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC, "-o", tmp,
                   *SOURCES]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            subprocess.run(cmd, check=True)
            os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build_library(force=True))
