"""Build the gemm_f16 shared library in-tree with nvcc for sm_103a.

Output: async_barrier_pipelined_gb300/_lib/libgemm_f16.so (git-ignored).
One translation unit, one -gencode, so a build takes seconds on either the
x86 build host or the aarch64 GPU host.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG_DIR, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libgemm_f16.so")

SOURCES = [os.path.join(CSRC, "gemm_f16.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, "ptx.cuh"), os.path.join(CSRC, "schedule.h"),
                     os.path.join(CSRC, "gemm_pair.cuh"), os.path.join(CSRC, "gemm_pair_wide.cuh"),
                     os.path.join(CSRC, "attn_f16.cuh"),
                     os.path.join(CSRC, "attn_pair.cuh"), os.path.join(INCLUDE, "gemm_f16.h"),
                     os.path.join(INCLUDE, "attn_f16.h")]

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: set NVCC or put the CUDA toolkit on PATH")


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if any source is newer than it; return its path."""
    os.makedirs(LIB_DIR, exist_ok=True)
    if not force and os.path.exists(LIB_PATH):
        lib_t = os.path.getmtime(LIB_PATH)
        if all(os.path.getmtime(f) <= lib_t for f in DEPENDS):
            return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc_path(), *ARCH_FLAGS, "-O3", "-std=c++17", "-lineinfo",
           "-Xcompiler", "-fPIC", "-shared", "-I", INCLUDE, *SOURCES, "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
