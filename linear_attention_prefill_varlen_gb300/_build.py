"""Builds the CUDA library in-tree with nvcc (sm_103a only)."""

from __future__ import annotations

import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
SRC = os.path.join(PKG_DIR, "csrc", "kda_conv.cu")
HEADER = os.path.join(ROOT, "include", "kda_conv.h")
LIB_PATH = os.path.join(PKG_DIR, "libkdaconv.so")

# No fast-math: the taps are explicit fmaf calls, divisions and expf stay IEEE
# unless the source asks otherwise, and denormals are kept.
NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libkdaconv.so")


def build(force: bool = False, extra_flags: list[str] | None = None, out: str = LIB_PATH) -> str:
    """Compiles csrc/kda_conv.cu into libkdaconv.so next to this file."""
    newest = max(os.path.getmtime(SRC), os.path.getmtime(HEADER), os.path.getmtime(__file__))
    if not force and os.path.exists(out) and os.path.getmtime(out) >= newest and not extra_flags:
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc_path(), *NVCC_FLAGS, *(extra_flags or []), "-I", os.path.join(ROOT, "include"),
           "-o", tmp, SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out
