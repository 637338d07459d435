"""ctypes binding of libdq4 (include/dq4.h): argument marshalling only.

Every step of the computation runs in the CUDA library.  PyTorch is used for
device memory and streams; there is no CPU path and no fallback: the first
use of the library (any call, or the ``lib`` attribute) raises ImportError if
libdq4.so has not been built.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .build import LIB_PATH

OUT_F16, OUT_BF16, OUT_F32 = 0, 1, 2
_DTYPE_CODE = {torch.float16: OUT_F16, torch.bfloat16: OUT_BF16, torch.float32: OUT_F32}
_CODE_DTYPE = {v: k for k, v in _DTYPE_CODE.items()}

STATUS_NAMES = {
    0: "DQ4_OK", 1: "DQ4_ERR_NULL", 2: "DQ4_ERR_N", 3: "DQ4_ERR_BLOCKSIZE",
    4: "DQ4_ERR_NESTED_BLOCKSIZE", 5: "DQ4_ERR_DTYPE", 6: "DQ4_ERR_ALIGN",
    7: "DQ4_ERR_DEVICE", 8: "DQ4_ERR_ARCH", 9: "DQ4_ERR_LAUNCH", 10: "DQ4_ERR_TOO_LARGE",
    11: "DQ4_ERR_CUBLAS",
}


class Dq4Error(RuntimeError):
    """A nonzero status from the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        L = get_lib()
        msg = L.dq4_status_string(status).decode()
        extra = ""
        if status in (7, 8, 9):
            extra = f" (cudaError_t {L.dq4_last_cuda_error()})"
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}{extra}")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libdq4.so is not built ({LIB_PATH}); build it with "
            "quantized_weight_dequantization_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    p, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    L.dq4_abi_version.argtypes = []
    L.dq4_abi_version.restype = ctypes.c_int
    L.dq4_nested.argtypes = [p, p, p, p, p, f32, i64, i32, i32, i32, p, p]
    L.dq4_nested.restype = ctypes.c_int
    L.dq4_nested_transposed.argtypes = [p, p, p, p, p, f32, i64, i64, i32, i32, i32, p, p]
    L.dq4_nested_transposed.restype = ctypes.c_int
    L.dq4.argtypes = [p, p, p, i64, i32, i32, p, p]
    L.dq4.restype = ctypes.c_int
    L.dq4_nested_unfused.argtypes = [p, p, p, p, p, f32, i64, i32, i32, i32, p, p, p]
    L.dq4_nested_unfused.restype = ctypes.c_int
    L.dq4_nested_unfused_static.argtypes = [p, p, p, p, p, f32, i64, i32, i32, i32, p, p]
    L.dq4_nested_unfused_static.restype = ctypes.c_int
    L.dq4_int8_correction_prep.argtypes = [p, p, p, p, i64, i64, i64, i64, p, p, p, p]
    L.dq4_int8_correction_prep.restype = ctypes.c_int
    L.dq4_nested_out_prod.argtypes = [p, p, p, p, p, f32, i64, i64, i32, i32, p, i64, p, p, i64,
                                      p, p]
    L.dq4_nested_out_prod.restype = ctypes.c_int
    L.dq4_nested_linear.argtypes = [p, i32, p, p, p, p, p, f32, i64, i64, i64, i32, i32, i32, p,
                                    p, i64, p, p]
    L.dq4_nested_linear.restype = ctypes.c_int
    L.dq4_nested_linear_workspace_bytes.argtypes = [i64, i64, i64]
    L.dq4_nested_linear_workspace_bytes.restype = ctypes.c_int64
    L.dq4_nested_out_prod_workspace_bytes.argtypes = [i64, i64, i64]
    L.dq4_nested_out_prod_workspace_bytes.restype = ctypes.c_int64
    L.dq4_nested_host.argtypes = [p, p, p, p, p, f32, i64, i32, i32, i32, p, p, i64, p]
    L.dq4_nested_host.restype = ctypes.c_int
    L.dq4_nested_host_scratch_bytes.argtypes = [i64, i32, i32, i32]
    L.dq4_nested_host_scratch_bytes.restype = ctypes.c_int64
    L.dq4_status_string.argtypes = [ctypes.c_int]
    L.dq4_status_string.restype = ctypes.c_char_p
    L.dq4_last_cuda_error.argtypes = []
    L.dq4_last_cuda_error.restype = ctypes.c_int
    return L


_LIB = None


def get_lib() -> ctypes.CDLL:
    """The loaded library (loaded on first use; raises ImportError if not built)."""
    global _LIB
    if _LIB is None:
        _LIB = _load()
    return _LIB


def __getattr__(name):
    if name == "lib":
        return get_lib()
    raise AttributeError(name)


# ------------------------------------------------------------- helpers
def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


_WORKSPACES = {}


def _linear_workspace(M: int, N: int, K: int, device, handle) -> torch.Tensor:
    """The cached zero-filled workspace of (device, stream), grown to this problem's size."""
    need = int(get_lib().dq4_nested_linear_workspace_bytes(M, N, K))
    key = (device.index, handle)
    ws = _WORKSPACES.get(key)
    if need <= 0:
        return ws if ws is not None else torch.empty(0, dtype=torch.uint8, device=device)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(need, dtype=torch.uint8, device=device)
        torch.cuda.synchronize(device)  # zero-filled before any stream uses it
        _WORKSPACES[key] = ws
    return ws


def _check(t: torch.Tensor, name: str, dtype: torch.dtype, numel: int, device) -> None:
    if t.device.type != "cuda":
        raise ValueError(f"{name}: must be a CUDA tensor (the library reads device memory)")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name}: expected a tensor on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.numel() < numel:
        raise ValueError(f"{name}: needs at least {numel} elements, has {t.numel()}")


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _out_tensor(out, out_dtype, n, device):
    if out is None:
        return torch.empty(n, dtype=out_dtype, device=device)
    if out.dtype not in _DTYPE_CODE:
        raise TypeError(f"out: unsupported dtype {out.dtype}")
    _check(out, "out", out.dtype, n, device)
    return out


def sizes(n: int, blocksize: int, nested_blocksize: int = 1):
    """(packed bytes, NB outer blocks, NG nested groups) of a problem of n values."""
    nb = -(-n // blocksize)
    return (n + 1) // 2, nb, -(-nb // nested_blocksize)


# ------------------------------------------------------------- the API
def dq4_nested(packed: torch.Tensor, scale_codes: torch.Tensor, nested_absmax: torch.Tensor,
               scale_codebook: torch.Tensor, value_codebook: torch.Tensor, offset: float,
               n: int, blocksize: int = 64, nested_blocksize: int = 256,
               out_dtype: torch.dtype = torch.float16, out: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    """Fused nested 4-bit dequantization (one launch); returns ``out`` (allocated if None).

    Issue #21 "Fuse nested scale reconstruction into SM103 4-bit
    dequantization", section "Proposed experiment".  All tensors live on one
    CUDA device; the call is asynchronous on ``stream`` (default: current).
    """
    device = packed.device
    npk, nb, ng = sizes(n, blocksize, nested_blocksize)
    _check(packed, "packed", torch.uint8, npk, device)
    _check(scale_codes, "scale_codes", torch.uint8, nb, device)
    _check(nested_absmax, "nested_absmax", torch.float32, ng, device)
    _check(scale_codebook, "scale_codebook", torch.float32, 256, device)
    _check(value_codebook, "value_codebook", torch.float32, 16, device)
    if out is not None:
        out_dtype = out.dtype
    if out_dtype not in _DTYPE_CODE:
        raise TypeError(f"out_dtype: unsupported {out_dtype}")
    res = _out_tensor(out, out_dtype, n, device)
    st = get_lib().dq4_nested(_ptr(packed), _ptr(scale_codes), _ptr(nested_absmax),
                        _ptr(scale_codebook), _ptr(value_codebook), float(offset), n,
                        blocksize, nested_blocksize, _DTYPE_CODE[out_dtype], _ptr(res),
                        _stream_handle(stream, device))
    if st:
        raise Dq4Error(st, "dq4_nested")
    return res


def _check_host(t: torch.Tensor, name: str, dtype: torch.dtype, numel: int) -> None:
    if t.device.type != "cpu":
        raise ValueError(f"{name}: must be a CPU tensor (this form copies host memory)")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.numel() < numel:
        raise ValueError(f"{name}: needs at least {numel} elements, has {t.numel()}")


_SCRATCH = {}


def dq4_nested_host(packed: torch.Tensor, scale_codes: torch.Tensor,
                    nested_absmax: torch.Tensor, scale_codebook: torch.Tensor,
                    value_codebook: torch.Tensor, offset: float, n: int, blocksize: int = 64,
                    nested_blocksize: int = 256, out_dtype: torch.dtype = torch.float16,
                    out: Optional[torch.Tensor] = None, device=None, stream=None,
                    scratch: Optional[torch.Tensor] = None) -> torch.Tensor:
    """dq4_nested's values from host (CPU) tensors into a host tensor, pipelined.

    Inputs and ``out`` are CPU tensors (page-locked for the copies to overlap;
    ``out`` is allocated pinned if None).  The work runs chunk by chunk on
    ``device``'s ``stream`` (default: the current ones); ``out`` is complete
    once the stream reaches the point after this call.  ``scratch`` is device
    memory; by default a cached buffer per (device, stream) is used.
    """
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else \
        torch.device(device)
    npk, nb, ng = sizes(n, blocksize, nested_blocksize)
    _check_host(packed, "packed", torch.uint8, npk)
    _check_host(scale_codes, "scale_codes", torch.uint8, nb)
    _check_host(nested_absmax, "nested_absmax", torch.float32, ng)
    _check_host(scale_codebook, "scale_codebook", torch.float32, 256)
    _check_host(value_codebook, "value_codebook", torch.float32, 16)
    if out is not None:
        out_dtype = out.dtype
    if out_dtype not in _DTYPE_CODE:
        raise TypeError(f"out_dtype: unsupported {out_dtype}")
    if out is None:
        out = torch.empty(n, dtype=out_dtype, pin_memory=True)
    _check_host(out, "out", out_dtype, n)
    handle = _stream_handle(stream, device)
    if scratch is None:
        need = int(get_lib().dq4_nested_host_scratch_bytes(n, blocksize, nested_blocksize,
                                                          _DTYPE_CODE[out_dtype]))
        key = (device.index, handle)
        scratch = _SCRATCH.get(key)
        if scratch is None or scratch.numel() < need:
            scratch = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
            _SCRATCH[key] = scratch
    elif scratch.device != device or scratch.dtype != torch.uint8:
        raise ValueError("scratch must be a uint8 tensor on the device")
    st = get_lib().dq4_nested_host(_ptr(packed), _ptr(scale_codes), _ptr(nested_absmax),
                                   _ptr(scale_codebook), _ptr(value_codebook), float(offset), n,
                                   blocksize, nested_blocksize, _DTYPE_CODE[out_dtype],
                                   _ptr(out), _ptr(scratch), scratch.numel(), handle)
    if st:
        raise Dq4Error(st, "dq4_nested_host")
    return out


def dq4_nested_transposed(packed: torch.Tensor, scale_codes: torch.Tensor,
                          nested_absmax: torch.Tensor, scale_codebook: torch.Tensor,
                          value_codebook: torch.Tensor, offset: float, rows: int, cols: int,
                          blocksize: int = 64, nested_blocksize: int = 256,
                          out_dtype: torch.dtype = torch.float16,
                          out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Fused nested dequantization of a rows x cols weight, written transposed.

    Returns ``out`` shaped (cols, rows): out[c, r] is the dequantized value
    (r, c).  Same arithmetic as :func:`dq4_nested` (issue #21, section
    "Correctness requirements": transposed output stays bitwise identical).
    """
    device = packed.device
    n = rows * cols
    npk, nb, ng = sizes(n, blocksize, nested_blocksize)
    _check(packed, "packed", torch.uint8, npk, device)
    _check(scale_codes, "scale_codes", torch.uint8, nb, device)
    _check(nested_absmax, "nested_absmax", torch.float32, ng, device)
    _check(scale_codebook, "scale_codebook", torch.float32, 256, device)
    _check(value_codebook, "value_codebook", torch.float32, 16, device)
    if out is not None:
        out_dtype = out.dtype
    if out_dtype not in _DTYPE_CODE:
        raise TypeError(f"out_dtype: unsupported {out_dtype}")
    res = _out_tensor(out, out_dtype, n, device)
    st = get_lib().dq4_nested_transposed(
        _ptr(packed), _ptr(scale_codes), _ptr(nested_absmax), _ptr(scale_codebook),
        _ptr(value_codebook), float(offset), rows, cols, blocksize, nested_blocksize,
        _DTYPE_CODE[out_dtype], _ptr(res), _stream_handle(stream, device))
    if st:
        raise Dq4Error(st, "dq4_nested_transposed")
    return res.view(cols, rows) if out is None else res


def dq4(packed: torch.Tensor, absmax: torch.Tensor, value_codebook: torch.Tensor, n: int,
        blocksize: int = 64, out_dtype: torch.dtype = torch.float16,
        out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Non-nested 4-bit dequantization with an FP32 absmax per block (one launch)."""
    device = packed.device
    npk, nb, _ = sizes(n, blocksize)
    _check(packed, "packed", torch.uint8, npk, device)
    _check(absmax, "absmax", torch.float32, nb, device)
    _check(value_codebook, "value_codebook", torch.float32, 16, device)
    if out is not None:
        out_dtype = out.dtype
    if out_dtype not in _DTYPE_CODE:
        raise TypeError(f"out_dtype: unsupported {out_dtype}")
    res = _out_tensor(out, out_dtype, n, device)
    st = get_lib().dq4(_ptr(packed), _ptr(absmax), _ptr(value_codebook), n, blocksize,
                 _DTYPE_CODE[out_dtype], _ptr(res), _stream_handle(stream, device))
    if st:
        raise Dq4Error(st, "dq4")
    return res


def dq4_nested_unfused(packed: torch.Tensor, scale_codes: torch.Tensor,
                       nested_absmax: torch.Tensor, scale_codebook: torch.Tensor,
                       value_codebook: torch.Tensor, offset: float, n: int, blocksize: int = 64,
                       nested_blocksize: int = 256, out_dtype: torch.dtype = torch.float16,
                       out: Optional[torch.Tensor] = None,
                       scale_scratch: Optional[torch.Tensor] = None, stream=None):
    """The unfused three-launch sequence; returns (out, scale_scratch)."""
    device = packed.device
    npk, nb, ng = sizes(n, blocksize, nested_blocksize)
    _check(packed, "packed", torch.uint8, npk, device)
    _check(scale_codes, "scale_codes", torch.uint8, nb, device)
    _check(nested_absmax, "nested_absmax", torch.float32, ng, device)
    _check(scale_codebook, "scale_codebook", torch.float32, 256, device)
    _check(value_codebook, "value_codebook", torch.float32, 16, device)
    if out is not None:
        out_dtype = out.dtype
    if out_dtype not in _DTYPE_CODE:
        raise TypeError(f"out_dtype: unsupported {out_dtype}")
    res = _out_tensor(out, out_dtype, n, device)
    if scale_scratch is None:
        scale_scratch = torch.empty(max(nb, 1), dtype=torch.float32, device=device)
    _check(scale_scratch, "scale_scratch", torch.float32, nb, device)
    st = get_lib().dq4_nested_unfused(_ptr(packed), _ptr(scale_codes), _ptr(nested_absmax),
                                _ptr(scale_codebook), _ptr(value_codebook), float(offset), n,
                                blocksize, nested_blocksize, _DTYPE_CODE[out_dtype], _ptr(res),
                                _ptr(scale_scratch), _stream_handle(stream, device))
    if st:
        raise Dq4Error(st, "dq4_nested_unfused")
    return res, scale_scratch


def dq4_nested_unfused_static(packed: torch.Tensor, scale_codes: torch.Tensor,
                              nested_absmax: torch.Tensor, scale_codebook: torch.Tensor,
                              value_codebook: torch.Tensor, offset: float, n: int,
                              blocksize: int = 64, nested_blocksize: int = 256,
                              out_dtype: torch.dtype = torch.float16,
                              out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The unfused sequence with the library's own static FP32 scratch.

    For callers that must not allocate device memory while they run (pass a
    preallocated ``out``; the call itself allocates nothing).  Limited to
    ceil(n / blocksize) <= 4,194,304 outer blocks.  Calls that overlap on
    the GPU share one scratch array and race: keep them on one stream.
    """
    device = packed.device
    npk, nb, ng = sizes(n, blocksize, nested_blocksize)
    _check(packed, "packed", torch.uint8, npk, device)
    _check(scale_codes, "scale_codes", torch.uint8, nb, device)
    _check(nested_absmax, "nested_absmax", torch.float32, ng, device)
    _check(scale_codebook, "scale_codebook", torch.float32, 256, device)
    _check(value_codebook, "value_codebook", torch.float32, 16, device)
    if out is not None:
        out_dtype = out.dtype
    if out_dtype not in _DTYPE_CODE:
        raise TypeError(f"out_dtype: unsupported {out_dtype}")
    res = _out_tensor(out, out_dtype, n, device)
    st = get_lib().dq4_nested_unfused_static(
        _ptr(packed), _ptr(scale_codes), _ptr(nested_absmax), _ptr(scale_codebook),
        _ptr(value_codebook), float(offset), n, blocksize, nested_blocksize,
        _DTYPE_CODE[out_dtype], _ptr(res), _stream_handle(stream, device))
    if st:
        raise Dq4Error(st, "dq4_nested_unfused_static")
    return res


def int8_correction_prep(A: torch.Tensor, CB: torch.Tensor, SCB: torch.Tensor,
                         cols: torch.Tensor, subA: Optional[torch.Tensor] = None,
                         subB: Optional[torch.Tensor] = None,
                         bad_cols: Optional[torch.Tensor] = None, stream=None):
    """LLM.int8 correction operands in one launch: returns (subA[M, L], subB[L, N]).

    "Fuse LLM.int8 correction operand preparation into one CUDA kernel"
    (bitsandbytes issue #16): subA = A[:, cols] (bit for bit); subB is the
    FP16 dequantization RN16(RN32(RN32(CB * SCB) * RN32(1/127))) of CB's
    columns ``cols``, transposed.  ``bad_cols`` (an int32 CUDA tensor of one
    element) counts indices outside [0, K).
    """
    if A.dim() != 2 or CB.dim() != 2:
        raise ValueError("A and CB must be 2-D")
    device = A.device
    M, K = A.shape
    N = CB.shape[0]
    if CB.shape[1] != K:
        raise ValueError(f"CB has {CB.shape[1]} columns, A has {K}")
    Lc = cols.numel()
    if A.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("A must be float16 or bfloat16")
    _check(A, "A", A.dtype, M * K, device)
    _check(CB, "CB", torch.int8, N * K, device)
    _check(SCB, "SCB", torch.float32, N, device)
    _check(cols, "cols", torch.int64, Lc, device)
    if subA is None:
        subA = torch.empty((M, Lc), dtype=A.dtype, device=device)
    if subB is None:
        subB = torch.empty((Lc, N), dtype=torch.float16, device=device)
    _check(subA, "subA", A.dtype, M * Lc, device)
    _check(subB, "subB", torch.float16, Lc * N, device)
    if bad_cols is not None:
        _check(bad_cols, "bad_cols", torch.int32, 1, device)
    st = get_lib().dq4_int8_correction_prep(
        _ptr(A), _ptr(CB), _ptr(SCB), _ptr(cols), M, N, K, Lc, _ptr(subA), _ptr(subB),
        _ptr(bad_cols), _stream_handle(stream, device))
    if st:
        raise Dq4Error(st, "dq4_int8_correction_prep")
    return subA, subB


# The largest workspace out_prod takes by default: the bound on the transient of "cuda:
# out_prod dequantizes a 2D weight in row blocks" (at most 256 MiB).
OUT_PROD_WORKSPACE_MAX = 256 << 20
_OUT_PROD_WORKSPACES = {}


def _out_prod_workspace(rows: int, cols: int, ncols: int, device, handle) -> torch.Tensor:
    """The cached partial-tile workspace of (device, stream), grown to this problem's size
    (capped at OUT_PROD_WORKSPACE_MAX; the library takes fewer row ranges when it is)."""
    need = min(int(get_lib().dq4_nested_out_prod_workspace_bytes(rows, cols, ncols)),
               OUT_PROD_WORKSPACE_MAX)
    key = (device.index, handle)
    ws = _OUT_PROD_WORKSPACES.get(key)
    if need <= 0:
        return ws if ws is not None else torch.empty(0, dtype=torch.float32, device=device)
    if ws is None or ws.numel() * 4 < need:
        ws = torch.empty((need + 3) // 4, dtype=torch.float32, device=device)
        _OUT_PROD_WORKSPACES[key] = ws
    return ws


def out_prod(packed: torch.Tensor, scale_codes: torch.Tensor, nested_absmax: torch.Tensor,
             scale_codebook: torch.Tensor, value_codebook: torch.Tensor, offset: float,
             rows: int, cols: int, G: torch.Tensor, blocksize: int = 64,
             nested_blocksize: int = 256, dst: Optional[torch.Tensor] = None,
             workspace: Optional[torch.Tensor] = None, bad: Optional[torch.Tensor] = None,
             stream=None) -> torch.Tensor:
    """dst = W^T G with W the rows x cols dequantized weight (FP32), decoded in row blocks
    inside a tcgen05 GEMM with FP32 accuracy.

    "cuda: out_prod dequantizes a 2D weight in row blocks" (llama.cpp pull
    request #4), section "What".  ``workspace`` (float32) holds the partial tiles
    of the row ranges the SMs share; by default a cached buffer per (device,
    stream) of at most 256 MiB is used, and an empty tensor runs one range
    straight into dst.  Returns dst (cols x ncols, FP32).
    """
    device = packed.device
    n = rows * cols
    npk, nb, ng = sizes(n, blocksize, nested_blocksize)
    _check(packed, "packed", torch.uint8, npk, device)
    _check(scale_codes, "scale_codes", torch.uint8, nb, device)
    _check(nested_absmax, "nested_absmax", torch.float32, ng, device)
    _check(scale_codebook, "scale_codebook", torch.float32, 256, device)
    _check(value_codebook, "value_codebook", torch.float32, 16, device)
    if G.dim() != 2 or G.shape[0] != rows:
        raise ValueError(f"G must be rows x ncols ({rows} x ...), got {tuple(G.shape)}")
    ncols = G.shape[1]
    _check(G, "G", torch.float32, rows * ncols, device)
    if dst is None:
        dst = torch.empty((cols, ncols), dtype=torch.float32, device=device)
    _check(dst, "dst", torch.float32, cols * ncols, device)
    if bad is not None:
        _check(bad, "bad", torch.int32, 1, device)
    handle = _stream_handle(stream, device)
    if workspace is None:
        workspace = _out_prod_workspace(rows, cols, ncols, device, handle)
    elif workspace.numel() > 0:
        _check(workspace, "workspace", torch.float32, 1, device)
    st = get_lib().dq4_nested_out_prod(
        _ptr(packed), _ptr(scale_codes), _ptr(nested_absmax), _ptr(scale_codebook),
        _ptr(value_codebook), float(offset), rows, cols, blocksize, nested_blocksize, _ptr(G),
        ncols, _ptr(dst), _ptr(workspace) if workspace.numel() > 0 else None,
        workspace.numel() * 4, _ptr(bad), handle)
    if st:
        raise Dq4Error(st, "dq4_nested_out_prod")
    return dst


def linear(X: torch.Tensor, packed: torch.Tensor, scale_codes: torch.Tensor,
           nested_absmax: torch.Tensor, scale_codebook: torch.Tensor,
           value_codebook: torch.Tensor, offset: float, N: int, blocksize: int = 64,
           nested_blocksize: int = 256, out_dtype: Optional[torch.dtype] = None,
           Y: Optional[torch.Tensor] = None, bad: Optional[torch.Tensor] = None,
           stream=None, workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Y = X W^T with W (N x K) given as nested 4-bit codes, decoded inside a tcgen05 GEMM.

    X is M x K (bfloat16 or float16); W's values are those dq4_nested gives
    for X's dtype.  The dequantize-plus-linear path of issue #21 without the
    materialised weight.  K must be a multiple of 64.

    ``workspace`` (uint8, zero-filled before first use) lets the SMs share the
    tiles' K ranges when there are fewer tiles than SMs; by default a cached
    buffer per (device, stream) is used, and an empty tensor disables it.
    """
    if X.dim() != 2:
        raise ValueError("X must be 2-D (M x K)")
    if X.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("X must be float16 or bfloat16")
    device = X.device
    M, K = X.shape
    npk, nb, ng = sizes(N * K, blocksize, nested_blocksize)
    _check(X, "X", X.dtype, M * K, device)
    _check(packed, "packed", torch.uint8, npk, device)
    _check(scale_codes, "scale_codes", torch.uint8, nb, device)
    _check(nested_absmax, "nested_absmax", torch.float32, ng, device)
    _check(scale_codebook, "scale_codebook", torch.float32, 256, device)
    _check(value_codebook, "value_codebook", torch.float32, 16, device)
    if Y is not None:
        out_dtype = Y.dtype
    out_dtype = out_dtype or X.dtype
    if out_dtype not in _DTYPE_CODE:
        raise TypeError(f"out_dtype: unsupported {out_dtype}")
    if Y is None:
        Y = torch.empty((M, N), dtype=out_dtype, device=device)
    _check(Y, "Y", out_dtype, M * N, device)
    if bad is not None:
        _check(bad, "bad", torch.int32, 1, device)
    handle = _stream_handle(stream, device)
    if workspace is None:
        workspace = _linear_workspace(M, N, K, device, handle)
    elif workspace.numel() > 0:
        if workspace.device != device or workspace.dtype != torch.uint8:
            raise ValueError("workspace must be a uint8 tensor on X's device")
    st = get_lib().dq4_nested_linear(
        _ptr(X), _DTYPE_CODE[X.dtype], _ptr(packed), _ptr(scale_codes), _ptr(nested_absmax),
        _ptr(scale_codebook), _ptr(value_codebook), float(offset), M, N, K, blocksize,
        nested_blocksize, _DTYPE_CODE[out_dtype], _ptr(Y),
        _ptr(workspace) if workspace.numel() > 0 else None, workspace.numel(), _ptr(bad),
        handle)
    if st:
        raise Dq4Error(st, "dq4_nested_linear")
    return Y
