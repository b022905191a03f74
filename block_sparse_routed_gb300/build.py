"""Builds the in-tree CUDA library ``_build/libsparse_attn.so`` for sm_103a.

nvcc only (no cmake): each translation unit is compiled in parallel, then
linked into one shared library with the CUDA runtime linked statically and
its symbols kept private.  Only the C-ABI entry points are exported.
"""

from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB_NAME = "libsparse_attn.so"
LIB_PATH = os.path.join(OUT, LIB_NAME)
SOURCES = ["api.cu", "plan_kernels.cu", "attn_kernel.cu", "plan_static.cu", "spark_reweight.cu", "reblock.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-lineinfo",
    "-O3",
    "-std=c++17",
    "-Xcompiler",
    "-fPIC,-fvisibility=hidden",
    "-I",
    os.path.join(ROOT, "include"),
    "-I",
    CSRC,
]


def find_nvcc() -> str:
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r


def build(verbose: bool = False, extra_flags=()) -> str:
    """Compile and link the library; return its path."""
    nvcc = find_nvcc()
    os.makedirs(OUT, exist_ok=True)
    objs = []
    cmds = []
    for src in SOURCES:
        obj = os.path.join(OUT, os.path.splitext(src)[0] + ".o")
        objs.append(obj)
        cmds.append([nvcc, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj])
    with ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        list(ex.map(lambda c: _run(c, verbose), cmds))
    tmp = LIB_PATH + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-Xlinker", "--exclude-libs,ALL"], verbose)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose=True))
