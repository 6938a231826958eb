"""Build the gemm_f16 shared library in-tree with nvcc for sm_103a.

Output: async_barrier_pipelined_gb300/_lib/libgemm_f16.so (git-ignored).
Three translation units (plan and shared host code, the GEMM kernels and
entry points, the attention kernels and entry points) are compiled in
parallel with one -gencode each and linked into one library, so a build
takes seconds on either the x86 build host or the aarch64 GPU host.
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

SOURCES = [os.path.join(CSRC, f) for f in ("plan.cu", "gemm_f16.cu", "attn_f16.cu")]
HEADERS = [os.path.join(CSRC, f) for f in ("host.h", "ptx.cuh", "schedule.h", "common.cuh",
                                            "gemm_pair.cuh", "gemm_quad.cuh", "attn_f16.cuh",
                                            "attn_pair.cuh")]
DEPENDS = SOURCES + HEADERS + [os.path.join(INCLUDE, "gemm_f16.h"),
                               os.path.join(INCLUDE, "attn_f16.h")]

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: set NVCC or put the CUDA toolkit on PATH")


def _compile_cmds(objs: list[str], verbose: bool) -> list[list[str]]:
    cmds = []
    for src, obj in zip(SOURCES, objs):
        cmd = [nvcc_path(), *ARCH_FLAGS, "-O3", "-std=c++17", "-lineinfo",
               "-Xcompiler", "-fPIC", "-I", INCLUDE, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        cmds.append(cmd)
    return cmds


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if any source is newer than it; return its path."""
    os.makedirs(LIB_DIR, exist_ok=True)
    if not force and os.path.exists(LIB_PATH):
        lib_t = os.path.getmtime(LIB_PATH)
        if all(os.path.getmtime(f) <= lib_t for f in DEPENDS):
            return LIB_PATH
    tag = f".tmp{os.getpid()}"
    objs = [os.path.join(LIB_DIR, os.path.basename(s)[:-3] + tag + ".o") for s in SOURCES]
    try:
        procs = [subprocess.Popen(c) for c in _compile_cmds(objs, verbose)]
        codes = [p.wait() for p in procs]
        if any(codes):
            raise subprocess.CalledProcessError(next(c for c in codes if c), "nvcc -c")
        tmp = LIB_PATH + tag
        subprocess.run([nvcc_path(), *ARCH_FLAGS, "-shared", *objs, "-o", tmp], check=True)
        os.replace(tmp, LIB_PATH)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
