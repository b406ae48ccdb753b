"""Build libmoe_mxfp4.so in-tree for sm_103a (nvcc cross-compiles without a GPU)."""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libmoe_mxfp4.so")
SRC = os.path.join(HERE, "csrc", "moe_mxfp4.cu")

NVCC_FLAGS = ["-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
              "-shared", "-Xcompiler", "-fPIC,-O2", "-cudart", "shared",
              "-I", os.path.join(ROOT, "include")]


def build(verbose_ptxas: bool = False, out: str = LIB, defines=()) -> str:
    """Compile the library to ``out``; ``defines`` are extra -D tuning knobs."""
    cmd = ["nvcc", *NVCC_FLAGS, *[f"-D{d}" for d in defines], "-o", out, SRC]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.check_call(cmd)
    return out


if __name__ == "__main__":
    build(verbose_ptxas="-v" in sys.argv)
