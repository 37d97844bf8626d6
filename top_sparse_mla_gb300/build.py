"""Compile the CUDA library (libdsa_sparse_attn.so) in-tree for sm_103a."""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
SOURCES = [os.path.join(PKG_DIR, "csrc", f) for f in ("dsa_sparse_attn.cu", "dsa_topk.cu", "dsa_kv_insert.cu")]
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libdsa_sparse_attn.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")


def build(verbose: bool = False, extra_flags=None) -> str:
    """Build the shared library if any source is newer than it; return its path."""
    deps = SOURCES + [os.path.join(PKG_DIR, "csrc", "ptx_sm103.cuh"), os.path.join(INCLUDE, "dsa_sparse_attn.h"),
                      os.path.join(INCLUDE, "dsa_topk.h"), os.path.join(INCLUDE, "dsa_kv_insert.h"),
            os.path.abspath(__file__)]
    if os.path.exists(LIB_PATH) and all(os.path.getmtime(LIB_PATH) >= os.path.getmtime(d) for d in deps):
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc_path(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-o", tmp, *SOURCES, *(extra_flags or [])]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose=True))
