"""Compile the CUDA library libdq4.so in-tree for sm_103a (nvcc, no cmake)."""

from __future__ import annotations

import concurrent.futures
import os
import subprocess
import sys
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
SOURCES = [os.path.join(CSRC, f) for f in
           ("flat.cu", "transposed.cu", "int8_prep.cu", "out_prod.cu", "linear.cu",
            "host_pipeline.cu", "host.cu")]
HEADERS = [os.path.join(ROOT, "include", "dq4.h"), os.path.join(CSRC, "common.cuh"),
           os.path.join(CSRC, "tcgen05.cuh"), os.path.join(CSRC, "tmap.cuh")]
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libdq4.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-fmad=false",            # no contraction anywhere (the kernels also use __fmul_rn/__fadd_rn)
    "-Xcompiler", "-fPIC",
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
    """Build libdq4.so (if stale) and return its path.

    The translation units compile in parallel (one nvcc each), then link into
    one shared library; ptxas's register report goes to ptxas.txt beside it.
    """
    dst = out or LIB_PATH
    if not force and not _stale(dst):
        return dst
    bdir = os.path.dirname(dst)
    os.makedirs(bdir, exist_ok=True)
    tag = f"{os.getpid()}"
    incs = ["-I", os.path.join(ROOT, "include"), "-I", CSRC]

    def compile_one(src):
        obj = os.path.join(bdir, f"{os.path.basename(src)}.{tag}.o")
        cmd = [nvcc(), *NVCC_FLAGS, *extra_flags, *incs, "-Xptxas", "-v", "-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, cmd, res

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    report = []
    failed = False
    for src, obj, cmd, res in results:
        report.append(" ".join(cmd) + "\n" + res.stdout + res.stderr)
        if res.returncode != 0:
            sys.stderr.write(res.stdout + res.stderr)
            failed = True
    objs = [obj for _, obj, _, _ in results]
    try:
        if failed:
            raise RuntimeError(f"nvcc failed building {dst}")
        tmp = f"{dst}.{tag}.tmp"
        link = [nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", *objs,
                "-o", tmp, "-ldl"]
        res = subprocess.run(link, capture_output=True, text=True)
        report.append(" ".join(link) + "\n" + res.stdout + res.stderr)
        if res.returncode != 0:
            sys.stderr.write(res.stdout + res.stderr)
            raise RuntimeError(f"link failed building {dst}")
        os.replace(tmp, dst)
    finally:
        with open(os.path.join(bdir, "ptxas.txt"), "w") as f:
            f.write("\n".join(report))
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    return dst


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
