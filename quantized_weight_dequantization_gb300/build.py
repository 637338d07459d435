"""Compile the CUDA library libdq4.so in-tree for sm_103a (nvcc, no cmake)."""

from __future__ import annotations

import os
import subprocess
import sys
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SOURCES = [os.path.join(PKG, "csrc", "dq4.cu")]
HEADERS = [os.path.join(ROOT, "include", "dq4.h")]
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libdq4.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-fmad=false",            # no contraction anywhere (the kernels also use __fmul_rn/__fadd_rn)
    "-Xcompiler", "-fPIC", "-shared",
    "-Xptxas", "-v",
]


def nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        path = os.path.join(cand, "bin", "nvcc") if cand else ""
        if path and os.path.exists(path):
            return path
    return "nvcc"


def _stale(dst: str) -> bool:
    if not os.path.exists(dst):
        return True
    t = os.path.getmtime(dst)
    return any(os.path.getmtime(s) > t for s in SOURCES + HEADERS + [__file__])


def build(force: bool = False, out: Optional[str] = None, extra_flags=()) -> str:
    """Build libdq4.so (if stale) and return its path.  ptxas's report goes to _build/."""
    dst = out or LIB_PATH
    if not force and not _stale(dst):
        return dst
    os.makedirs(os.path.dirname(dst), exist_ok=True)
    tmp = f"{dst}.{os.getpid()}.tmp"
    cmd = [nvcc(), *NVCC_FLAGS, *extra_flags, "-I", os.path.join(ROOT, "include"),
           *SOURCES, "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(os.path.dirname(dst), "ptxas.txt"), "w") as f:
        f.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError(f"nvcc failed ({res.returncode}) building {dst}")
    os.replace(tmp, dst)
    return dst


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
