"""Build ``libtp_b300.so`` in-tree with nvcc for sm_103a (B300).

    python -m tensor_sharded_linear_02_b300.build [--force] [--verbose]

The library is csrc/tp_api.cu (which includes the kernel headers) plus
csrc/tp_static_ws.cu, linked against the static CUDA runtime so that the
only runtime dependency is the driver.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libtp_b300.so")
MAIN = os.path.join(HERE, "csrc", "tp_api.cu")
STATIC_WS = os.path.join(HERE, "csrc", "tp_static_ws.cu")

NVCC_FLAGS = [
    "-O3", "-std=c++17",
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo",
    "-Xcompiler", "-fPIC", "-shared",
    "-cudart", "static",
]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return ([MAIN, STATIC_WS] + glob.glob(os.path.join(HERE, "csrc", "*.cuh"))
            + [os.path.join(ROOT, "include", "tp.h")])


def build(force: bool = False, verbose: bool = False) -> str:
    stale = not os.path.exists(LIB) or any(
        os.path.getmtime(s) > os.path.getmtime(LIB) for s in _sources())
    if not (force or stale):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ([_nvcc()] + NVCC_FLAGS + (["-Xptxas", "-v"] if verbose else [])
           + [MAIN, STATIC_WS, "-o", tmp])
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
