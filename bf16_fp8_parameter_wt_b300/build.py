"""Build libwt.so in-tree with nvcc for sm_103a.

IEEE division and denormals stay on (-prec-div=true -ftz=false): the
kernels' results must be bit-exact, and block scales can be subnormal.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
SOURCES = ["api.cpp", "plan.cpp", "tmap.cpp", "prep_kernel.cu", "token_kernel.cu", "counters.cu", "noalloc.cu",
           "codec_sweep.cu"]
HEADERS = ["plan.h", "codec.cuh", "ptx.cuh"]
LIB = os.path.join(HERE, "libwt.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc_cmd(out: str, verbose: bool = False) -> list:
    cmd = ["nvcc", ARCH, "-lineinfo", "-O3", "-std=c++17", "-prec-div=true", "-ftz=false",
           "-Xcompiler", "-fPIC,-O2,-Wall", "-shared", "-cudart", "static",
           f"-I{os.path.join(ROOT, 'include')}", "-o", out]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    return cmd + [os.path.join(CSRC, s) for s in SOURCES]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(ROOT, "include", "wt.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if force or _stale():
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(nvcc_cmd(tmp, verbose))
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose=True)
