"""CPU oracle for nested 4-bit dequantization: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports, links or runs it, and it shares no code with
the product: the scalar C file ``dq4_oracle.c`` is built here with gcc, and
``checker.py`` is a second, independent numpy/torch-CPU implementation.

Method: "Fuse nested scale reconstruction into SM103 4-bit dequantization"
(bitsandbytes issue #21), sections "Proposed experiment" (the two formulas)
and "Correctness requirements" (separately rounded FP32 multiply and add,
bitwise identity with the unfused sequence of section "Problem").
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dq4_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle_dq4.so")

# -ffp-contract=off: the scale's multiply and add must round separately.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-Wall", "-Wextra"]

OUT_CODES = {"f16": 0, "bf16": 1, "f32": 2}
OUT_NP = {"f16": np.uint16, "bf16": np.uint16, "f32": np.float32}

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def build(force: bool = False, src: str = _SRC, dst: str = _LIB_PATH,
          extra_flags: Optional[list] = None) -> str:
    """Compile the C oracle into a shared library (gcc); return its path."""
    if not force and os.path.exists(dst) and os.path.getmtime(dst) >= os.path.getmtime(src):
        return dst
    os.makedirs(os.path.dirname(dst), exist_ok=True)
    tmp = f"{dst}.{os.getpid()}.tmp"
    cmd = ["gcc", *CFLAGS, *(extra_flags or []), src, "-o", tmp]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, dst)
    return dst


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    p, i64, f32, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
    lib.oracle_f32_to_f16.argtypes = [f32]
    lib.oracle_f32_to_f16.restype = ctypes.c_uint16
    lib.oracle_f32_to_bf16.argtypes = [f32]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_f32_to_f16_array.argtypes = [p, p, i64]
    lib.oracle_f32_to_bf16_array.argtypes = [p, p, i64]
    lib.oracle_convert_bit_range.argtypes = [ctypes.c_uint32, i64, i32, p]
    lib.oracle_nested_scale.argtypes = [ctypes.c_uint8, f32, p, f32]
    lib.oracle_nested_scale.restype = f32
    lib.oracle_dq4_nested.argtypes = [p, p, p, p, p, f32, i64, i64, i64, i32, p]
    lib.oracle_dq4.argtypes = [p, p, p, i64, i64, i32, p]
    lib.oracle_dq4_nested_transposed.argtypes = [p, p, p, p, p, f32, i64, i64, i64, i64, i32, p]
    lib.oracle_nested_scales.argtypes = [p, p, p, f32, i64, i64, p]
    lib.oracle_int8_correction_prep.argtypes = [p, p, p, p, i64, i64, i64, i64, p, p]
    for name in ("oracle_f32_to_f16_array", "oracle_f32_to_bf16_array",
                 "oracle_convert_bit_range", "oracle_dq4_nested", "oracle_dq4",
                 "oracle_nested_scales", "oracle_dq4_nested_transposed",
                 "oracle_int8_correction_prep"):
        getattr(lib, name).restype = None
    return lib


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """The oracle library (built on first use)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ----------------------------------------------------------------- method
def dq4_nested(problem, out: str = "f16", threads: int = 1, lib=None) -> np.ndarray:
    """Dequantize ``problem`` (a dq4_inputs.Problem); uint16 bits or float32 values.

    With ``threads > 1`` the flat range is cut at nested-group boundaries
    (multiples of blocksize * nested_blocksize values) and the same scalar
    routine runs on each piece in its own thread; the arithmetic is unchanged.
    """
    lib = lib or load()
    p = problem
    res = np.empty(p.n, dtype=OUT_NP[out])
    itemsize = res.itemsize
    unit = p.blocksize * p.nested_blocksize
    units = -(-p.n // unit)
    threads = max(1, min(threads, units))
    bounds = [min(p.n, (units * t // threads) * unit) for t in range(threads + 1)]

    def run(lo, hi):
        if hi <= lo:
            return
        lib.oracle_dq4_nested(
            _ptr(p.packed) + lo // 2, _ptr(p.scale_codes) + lo // p.blocksize,
            _ptr(p.nested_absmax) + 4 * (lo // unit), _ptr(p.scale_codebook),
            _ptr(p.value_codebook), float(p.offset), hi - lo, p.blocksize,
            p.nested_blocksize, OUT_CODES[out], _ptr(res) + itemsize * lo)

    if threads == 1:
        run(0, p.n)
    else:
        ts = [threading.Thread(target=run, args=(bounds[t], bounds[t + 1]))
              for t in range(threads)]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
    return res


def dq4_nested_transposed(problem, rows: int, cols: int, out: str = "f16",
                          threads: int = 1, lib=None) -> np.ndarray:
    """Dequantize ``problem`` as a rows x cols weight and return W^T flat (cols x rows).

    With ``threads > 1`` the threaded flat oracle runs and numpy's transpose
    (a library primitive) is the last step; the arithmetic is unchanged.
    """
    lib = lib or load()
    p = problem
    assert rows * cols == p.n
    if threads <= 1:
        res = np.empty(p.n, dtype=OUT_NP[out])
        lib.oracle_dq4_nested_transposed(
            _ptr(p.packed), _ptr(p.scale_codes), _ptr(p.nested_absmax), _ptr(p.scale_codebook),
            _ptr(p.value_codebook), float(p.offset), rows, cols, p.blocksize,
            p.nested_blocksize, OUT_CODES[out], _ptr(res))
        return res
    flat = dq4_nested(p, out, threads=threads, lib=lib).reshape(rows, cols)
    return np.ascontiguousarray(flat.T).reshape(-1)


def dq4(packed: np.ndarray, absmax: np.ndarray, value_codebook: np.ndarray, n: int,
        blocksize: int, out: str = "f16", lib=None) -> np.ndarray:
    """Non-nested dequantization with a given FP32 absmax per block."""
    lib = lib or load()
    res = np.empty(n, dtype=OUT_NP[out])
    lib.oracle_dq4(_ptr(packed), _ptr(absmax), _ptr(value_codebook), n, blocksize,
                   OUT_CODES[out], _ptr(res))
    return res


def nested_scales(problem, lib=None) -> np.ndarray:
    """FP32 per-block scales of the unfused sequence (steps 1 and 2)."""
    lib = lib or load()
    p = problem
    res = np.empty(p.nblocks, dtype=np.float32)
    lib.oracle_nested_scales(_ptr(p.scale_codes), _ptr(p.nested_absmax),
                             _ptr(p.scale_codebook), float(p.offset), p.nblocks,
                             p.nested_blocksize, _ptr(res))
    return res


def nested_scale(code: int, absmax: float, scale_codebook: np.ndarray, offset: float,
                 lib=None) -> np.float32:
    lib = lib or load()
    return np.float32(lib.oracle_nested_scale(code, float(np.float32(absmax)),
                                              _ptr(scale_codebook), float(np.float32(offset))))


def f32_to_f16_bits(x: np.ndarray, lib=None) -> np.ndarray:
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib.oracle_f32_to_f16_array(_ptr(x), _ptr(y), x.size)
    return y


def f32_to_bf16_bits(x: np.ndarray, lib=None) -> np.ndarray:
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib.oracle_f32_to_bf16_array(_ptr(x), _ptr(y), x.size)
    return y


def convert_bit_range(first: int, count: int, to_bf16: bool, lib=None) -> np.ndarray:
    """Convert every binary32 bit pattern in [first, first+count)."""
    lib = lib or load()
    y = np.empty(count, dtype=np.uint16)
    lib.oracle_convert_bit_range(first, count, int(to_bf16), _ptr(y))
    return y


def int8_correction_prep(A_bits: np.ndarray, CB: np.ndarray, SCB: np.ndarray, cols: np.ndarray,
                         lib=None):
    """LLM.int8 correction operands (issue #16): (subA[M, L], subB[L, N]) as uint16 bits."""
    lib = lib or load()
    M, K = A_bits.shape
    N = CB.shape[0]
    L = cols.size
    A_bits = np.ascontiguousarray(A_bits, dtype=np.uint16)
    CB = np.ascontiguousarray(CB, dtype=np.int8)
    SCB = np.ascontiguousarray(SCB, dtype=np.float32)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    assert CB.shape[1] == K and SCB.size == N
    assert L == 0 or (cols.min() >= 0 and cols.max() < K)
    subA = np.empty((M, L), dtype=np.uint16)
    subB = np.empty((L, N), dtype=np.uint16)
    if L:
        lib.oracle_int8_correction_prep(_ptr(A_bits), _ptr(CB), _ptr(SCB), _ptr(cols), M, N, K,
                                        L, _ptr(subA), _ptr(subB))
    return subA, subB


def out_prod(problem, rows: int, cols: int, G: np.ndarray, threads: int = 8, lib=None):
    """dst = W^T G in float64: W is the oracle's FP32 dequantization (rows x cols).

    The FP32 values of W are exact in float64; numpy's float64 matmul (a
    library primitive) is the contraction.  Reading: "cuda: out_prod
    dequantizes a 2D weight in row blocks" (llama.cpp pull request #4),
    section "What": out_prod sums over the weight's rows.
    """
    w = dq4_nested(problem, "f32", threads=threads, lib=lib).reshape(rows, cols)
    return w.astype(np.float64).T @ np.asarray(G, dtype=np.float64)


def linear(problem, X_bits: np.ndarray, in_dtype: str, N: int, K: int, threads: int = 8,
           lib=None) -> np.ndarray:
    """Y = X W^T in float64: W is the oracle's dequantization to ``in_dtype`` (N x K).

    X_bits holds X's raw 16-bit values (M x K).  Both operands are exact in
    float64; numpy's float64 matmul (a library primitive) is the contraction.
    """
    w = dq4_nested(problem, in_dtype, threads=threads, lib=lib).reshape(N, K)
    return _bits16_to_f64(X_bits, in_dtype) @ _bits16_to_f64(w, in_dtype).T


def _bits16_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
