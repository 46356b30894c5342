"""Build the sm_103a shared library ``libttt_mlp.so`` in-tree with nvcc.

Usage: ``python -m chunk_wise_weight_ttt_b300.build`` (or call ``build()``).
nvcc cross-compiles without a GPU present.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB = os.path.join(PKG, "libttt_mlp.so")
SRC = os.path.join(PKG, "csrc", "ttt_mlp.cu")
DEPS = [os.path.join(PKG, "csrc", n) for n in ("sm100_ptx.cuh", "tc_gemm.cuh", "simt_kernels.cuh")]
HDR = os.path.join(ROOT, "include", "ttt_mlp.h")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libttt_mlp.so")
    return exe


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in [SRC, HDR, *DEPS])


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(nvcc())), "lib64")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           "-cudart", "shared", f"-I{os.path.join(ROOT, 'include')}", "-o", LIB + ".tmp", SRC,
           "-Xlinker", f"-rpath,{cuda_lib}"]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed ({r.returncode}):\n{r.stdout}\n{r.stderr}")
    if verbose:
        sys.stderr.write(r.stderr)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
