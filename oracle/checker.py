"""Second, independent CPU implementation of nested 4-bit dequantization.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Vectorised numpy /
torch-CPU: float32 ufuncs, each a single IEEE operation, so nothing is ever
contracted into an FMA; the output conversions are numpy's float16 cast and
torch's bfloat16 cast, both round-to-nearest-even.  It shares no code with the
C oracle, so agreement between the two pins each against the other.

Formulas: "Fuse nested scale reconstruction into SM103 4-bit dequantization"
(bitsandbytes issue #21), section "Proposed experiment"; rounding order from
section "Correctness requirements".
"""

from __future__ import annotations

import numpy as np
import torch


def unpack_nibbles(packed: np.ndarray, n: int) -> np.ndarray:
    """Codes of values 0..n-1: even index from the high nibble, odd from the low."""
    codes = np.empty(2 * packed.size, dtype=np.uint8)
    codes[0::2] = packed >> 4
    codes[1::2] = packed & 0x0F
    return codes[:n]


def to_out_bits(v: np.ndarray, out: str) -> np.ndarray:
    """float32 values -> output (raw uint16 bits for f16/bf16, float32 for f32)."""
    if out == "f16":
        return v.astype(np.float16).view(np.uint16)
    if out == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(v)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16)
    if out == "f32":
        return v.astype(np.float32, copy=True)
    raise ValueError(out)


def block_scales(scale_codes, nested_absmax, scale_codebook, offset, nested_blocksize):
    """Per-block FP32 scale: the product and the sum are two separate float32 ops."""
    b = np.arange(scale_codes.size)
    prod = scale_codebook[scale_codes] * nested_absmax[b // nested_blocksize]
    assert prod.dtype == np.float32
    return prod + np.float32(offset)


def dq4_from_scales(packed, scales, value_codebook, n, blocksize, out):
    v = value_codebook[unpack_nibbles(packed, n)] * np.repeat(scales, blocksize)[:n]
    assert v.dtype == np.float32
    return to_out_bits(v, out)


def dq4_nested(problem, out: str = "f16", chunk_values: int = 1 << 24) -> np.ndarray:
    """The whole problem, processed in nested-group-aligned chunks to bound memory."""
    p = problem
    unit = p.blocksize * p.nested_blocksize
    chunk = max(unit, (chunk_values // unit) * unit)
    parts = []
    for lo in range(0, p.n, chunk):
        hi = min(p.n, lo + chunk)
        b0, b1 = lo // p.blocksize, -(-hi // p.blocksize)
        g0, g1 = lo // unit, -(-hi // unit)
        s = block_scales(p.scale_codes[b0:b1], p.nested_absmax[g0:g1], p.scale_codebook,
                         p.offset, p.nested_blocksize)
        parts.append(dq4_from_scales(p.packed[lo // 2:(hi + 1) // 2], s, p.value_codebook,
                                     hi - lo, p.blocksize, out))
    if not parts:
        return to_out_bits(np.empty(0, dtype=np.float32), out)
    return np.concatenate(parts)


def int8_correction_prep(A_bits, CB, SCB, cols):
    """Second implementation of the LLM.int8 correction operands (issue #16).

    subA is a numpy fancy-index gather of the raw bits; subB is two float32
    ufunc multiplies (CB * SCB, then * float32(1)/float32(127)) and numpy's
    float16 cast, transposed.
    """
    subA = np.ascontiguousarray(A_bits[:, cols])
    recip = np.float32(1) / np.float32(127)
    t1 = CB[:, cols].astype(np.float32) * SCB.astype(np.float32)[:, None]
    t2 = t1 * recip
    assert t2.dtype == np.float32
    with np.errstate(over="ignore"):
        subB = np.ascontiguousarray(t2.T.astype(np.float16).view(np.uint16))
    return subA, subB
