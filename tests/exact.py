"""Exact rational arithmetic with explicit IEEE-754 rounding, for pinning the oracle.

A third, independent way to evaluate the method: every operation is done
exactly with ``fractions.Fraction`` and then rounded to the target format by
round-to-nearest-even from the textbook definition (quantum 2^Q with
Q = max(floor(log2|x|), emin) - (p - 1); ties to the even integer multiple;
a result of 2^(emax + 1) or more overflows to infinity).  Signed zeros follow
IEEE-754: a product's zero takes the XOR of the signs; an exact-zero sum is
+0 unless both addends are -0.

It shares no code with ``oracle/`` (bit manipulation in C, float32 ufuncs in
numpy) or with the CUDA path.
"""

from __future__ import annotations

import math
from fractions import Fraction
from typing import NamedTuple

import numpy as np
import torch

# (p = significand bits incl. the hidden one, emin, emax)
F32 = (24, -126, 127)
F16 = (11, -14, 15)
BF16 = (8, -126, 127)


class Val(NamedTuple):
    """An exactly known floating value: magnitude-with-sign, plus the sign of a zero."""

    q: Fraction          # exact value (0 for zeros)
    neg: bool            # sign bit
    inf: bool = False


def from_f32(x) -> Val:
    x = float(np.float32(x))
    assert math.isfinite(x)
    return Val(Fraction(x), math.copysign(1.0, x) < 0)


def _floor_log2(a: Fraction) -> int:
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def round_to(q: Fraction, neg: bool, fmt) -> Val:
    """Round the exact value q to format fmt (RNE). ``neg`` gives the sign of a zero result."""
    p, emin, emax = fmt
    if q == 0:
        return Val(Fraction(0), neg)
    sign = q < 0
    a = -q if sign else q
    e = _floor_log2(a)
    quantum = Fraction(2) ** (max(e, emin) - (p - 1))
    scaled = a / quantum
    r = scaled.numerator // scaled.denominator
    rem = scaled - r
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and r % 2 == 1):
        r += 1
    mag = r * quantum
    if mag >= Fraction(2) ** (emax + 1):
        return Val(Fraction(0), sign, inf=True)
    return Val(-mag if sign else mag, sign)


def mul(a: Val, b: Val, fmt=F32) -> Val:
    return round_to(a.q * b.q, a.neg != b.neg, fmt)


def add(a: Val, b: Val, fmt=F32) -> Val:
    exact = a.q + b.q
    return round_to(exact, a.neg and b.neg, fmt)


def to_float(v: Val) -> float:
    if v.inf:
        return -math.inf if v.neg else math.inf
    if v.q == 0:
        return -0.0 if v.neg else 0.0
    return float(v.q)  # exact: every value here is representable in binary64


def f32_value(v: Val) -> np.float32:
    return np.float32(to_float(v))


def f16_bits(v: Val) -> int:
    """Bits of an already-rounded FP16 value (the cast is exact)."""
    return int(np.array(to_float(v), dtype=np.float64).astype(np.float16).view(np.uint16))


def bf16_bits(v: Val) -> int:
    """Bits of an already-rounded BF16 value (the cast is exact)."""
    t = torch.tensor([to_float(v)], dtype=torch.float64).to(torch.bfloat16)
    return int(t.view(torch.int16).item()) & 0xFFFF


def f32_bits(v: Val) -> int:
    return int(np.array([to_float(v)], dtype=np.float32).view(np.uint32)[0])


def nested_scale(scb_k, absmax_g, offset) -> Val:
    """scale = RN32(RN32(scb[k] * A[g]) + offset)."""
    return add(mul(from_f32(scb_k), from_f32(absmax_g)), from_f32(offset))


def fma_scale(scb_k, absmax_g, offset) -> Val:
    """The contracted form RN32(scb[k] * A[g] + offset) with a single rounding."""
    a, b, c = from_f32(scb_k), from_f32(absmax_g), from_f32(offset)
    prod = a.q * b.q
    return round_to(prod + c.q, (a.neg != b.neg) and c.neg, F32)


def output_bits(v32: Val, out: str) -> int:
    """The stored output (as raw bits) for an FP32 value v32."""
    if out == "f16":
        return f16_bits(round_to(v32.q, v32.neg, F16))
    if out == "bf16":
        return bf16_bits(round_to(v32.q, v32.neg, BF16))
    return f32_bits(v32)


def dequantize(problem, outs=("f16", "bf16", "f32")):
    """Value-by-value exact evaluation of a whole (small) problem.

    Returns {out: list of output bits}.  Results are memoised per
    (nibble, scale code, nested group), which leaves the arithmetic unchanged.
    """
    p = problem
    memo = {}
    res = {o: [] for o in outs}
    for i in range(p.n):
        byte = int(p.packed[i // 2])
        nib = (byte >> 4) if i % 2 == 0 else (byte & 0xF)
        b = i // p.blocksize
        g = b // p.nested_blocksize
        key = (nib, int(p.scale_codes[b]), g)
        if key not in memo:
            s = nested_scale(p.scale_codebook[key[1]], p.nested_absmax[g], p.offset)
            v = mul(from_f32(p.value_codebook[nib]), s)
            memo[key] = {o: output_bits(v, o) for o in outs}
        for o in outs:
            res[o].append(memo[key][o])
    return res
