"""Builds the CUDA library ``lib/librlk_logp.so`` in-tree with nvcc for sm_103a."""

from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
SOURCES = [os.path.join(CSRC, f) for f in ("rlk_logp.cu", "rlk_shard.cu", "rlk_grad.cu", "rlk_noalloc.cu",
                                          "rlk_linear.cu", "rlk_norm.cu", "rlk_host_io.cu")]
HEADERS = [os.path.join(CSRC, "rlk_device.cuh"), os.path.join(CSRC, "rlk_host.h")]
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIB_DIR, "librlk_logp.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librlk_logp.so")


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    lib_t = os.path.getmtime(LIB)
    deps = [*SOURCES, *HEADERS, os.path.join(INCLUDE, "rlk_logp.h"), os.path.join(INCLUDE, "rlk_norm.h")]
    return any(os.path.getmtime(d) > lib_t for d in deps)


def build_library(force: bool = False, verbose: bool = False) -> str:
    if not force and not needs_build():
        return LIB
    os.makedirs(LIB_DIR, exist_ok=True)
    tmp = LIB + ".tmp"
    # one nvcc call; --threads compiles the translation units in parallel
    cmd = [nvcc_path(), *NVCC_FLAGS, "--threads", "0", "-I", INCLUDE, "-o", tmp, *SOURCES]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
