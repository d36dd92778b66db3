"""Builds libmbglu.so in-tree with nvcc for sm_103a (GB300).

No fast math (DeepSpeed PR #9057 "Changes" removed --use_fast_math from the
fused-GLU build): expf and division keep their IEEE-accurate forms.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libmbglu.so")
SOURCES = [os.path.join(HERE, "csrc", "mbglu_api.cu")]
DEPS = SOURCES + [os.path.join(HERE, "csrc", f) for f in ("glu_kernels.cuh", "glu_backward.cuh", "glu_tc.cuh",
                                                         "glu_slice.cuh", "tcgen05.cuh", "ptx.cuh")] + \
    [os.path.join(ROOT, "include", "mbglu.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
    # share the process's CUDA runtime (the one torch loads), so the current
    # device and streams are one state; rpath for standalone C callers
    "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64",
    "-I", os.path.join(ROOT, "include"),
]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def needs_build(out: str = LIB) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(f) > t for f in DEPS)


def build(out: str = LIB, verbose: bool = False, extra=()) -> str:
    cmd = [nvcc(), *NVCC_FLAGS, *extra, "-o", out, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    return out


if __name__ == "__main__":
    build(verbose="-v" in sys.argv)
    print(LIB)
