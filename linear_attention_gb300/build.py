"""Builds the CUDA library in-tree with nvcc (sm_103a only)."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB_DIR = os.path.join(HERE, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libbased_gb300.so")
SOURCES = [os.path.join(CSRC, "based_fwd.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "based_kernels.cuh"), os.path.join(CSRC, "sm103_ptx.cuh"),
                  os.path.join(CSRC, "based_plan.h"),
                  os.path.join(ROOT, "include", "based.h")]
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared", "-Xcompiler", "-fvisibility=hidden"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the shared library if it is missing or older than any of its sources."""
    os.makedirs(LIB_DIR, exist_ok=True)
    if not force and os.path.exists(LIB_PATH):
        t = os.path.getmtime(LIB_PATH)
        if all(os.path.getmtime(p) <= t for p in DEPS):
            return LIB_PATH
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc()] + NVCC_FLAGS + SOURCES + ["-o", tmp]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
