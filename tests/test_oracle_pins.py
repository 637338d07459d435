"""Pins of the CPU oracle against what the method and IEEE-754 fix (no GPU).

Method: "Fuse nested scale reconstruction into SM103 4-bit dequantization"
(bitsandbytes issue #21): section "Proposed experiment" gives the two
formulas; section "Correctness requirements" asks for bitwise identity over
NF4/FP4, FP16/BF16/FP32, block sizes 32..4096, odd lengths and partial blocks
and groups, both offset signs, every scale code and every 4-bit code, with
the FP32 multiply and add rounded separately.

Each pin is independent of the oracle's own code: hand-worked closed forms
(tests/golden), exact rational arithmetic (tests/exact.py), torch/numpy
converters, numpy float32 scalar arithmetic, and algebraic special cases.
"""

import json
import os
import threading

import numpy as np
import pytest
import torch

import dq4_inputs as gen
import oracle
import oracle.checker as checker
from tests import exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")
OUTS = ("f16", "bf16", "f32")


def _u32(h):
    return np.array([int(h, 16)], dtype=np.uint32).view(np.float32)[0]


def _hand_problem(case):
    """The one-block problem a golden case describes."""
    scb = gen.scale_codebook().copy()
    scb[0] = _u32(case["scale_codebook_entry"])
    if "value_codebook" in case:
        vcb = (np.arange(16, dtype=np.float32) / np.float32(16))
        packed = np.array(case["packed"], dtype=np.uint8)
        n = case["n"]
    else:
        vcb = gen.nf4_style_codebook().copy()
        vcb[3] = _u32(case["value_codebook_entry"])
        packed = np.full(16, 0x33, dtype=np.uint8)
        n = 32
    return gen.Problem(packed=packed, scale_codes=np.zeros(1, dtype=np.uint8),
                       nested_absmax=np.array([_u32(case["nested_absmax"])], dtype=np.float32),
                       scale_codebook=scb, value_codebook=vcb.astype(np.float32),
                       offset=_u32(case["offset"]), n=n, blocksize=32, nested_blocksize=256)


def _bits(arr, out):
    return [int(x) for x in (arr.view(np.uint32) if out == "f32" else arr)]


def _load_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _load_cases(), ids=lambda c: c["name"])
def test_hand_worked_golden(case):
    p = _hand_problem(case)
    ex = exact.dequantize(p)
    for out in OUTS:
        got = _bits(oracle.dq4_nested(p, out), out)
        if "expected_values" in case:
            want = [int(h, 16) for h in case["expected_values"][out]]
        else:
            want = [int(case["expected"][out], 16)] * p.n
        assert got == want, (case["name"], out, [hex(x) for x in got[:4]])
        assert ex[out] == want, (case["name"], out, "exact evaluation disagrees with fixture")
    if "expected" in case:
        s = oracle.nested_scale(0, p.nested_absmax[0], p.scale_codebook, p.offset)
        assert hex(int(np.array([s]).view(np.uint32)[0])) == hex(int(case["expected"]["scale"], 16))


# ----------------------------------------------------------- conversions
def _torch_bits(x: np.ndarray, dtype) -> np.ndarray:
    return torch.from_numpy(x).to(dtype).view(torch.int16).numpy().view(np.uint16)


def _exhaustive(to_bf16: bool):
    chunk = 1 << 24
    mismatches = []
    lock = threading.Lock()

    def work(first):
        y = oracle.convert_bit_range(first, chunk, to_bf16)
        x = np.arange(first, first + chunk, dtype=np.uint32).view(np.float32)
        ref = _torch_bits(x, torch.bfloat16 if to_bf16 else torch.float16)
        nan_in = np.isnan(x)
        exp_mask = 0x7F80 if to_bf16 else 0x7C00
        man_mask = 0x007F if to_bf16 else 0x03FF
        ok_nan = ((y[nan_in] & exp_mask) == exp_mask) & ((y[nan_in] & man_mask) != 0)
        bad = np.flatnonzero((y != ref) & ~nan_in)
        with lock:
            if bad.size or not ok_nan.all():
                mismatches.append((first, bad[:4], int((~ok_nan).sum())))

    firsts = list(range(0, 1 << 32, chunk))
    threads = min(8, os.cpu_count() or 1)
    for k in range(0, len(firsts), threads):
        ts = [threading.Thread(target=work, args=(f,)) for f in firsts[k:k + threads]]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
    assert not mismatches, mismatches[:3]


def test_f16_converter_exhaustive_vs_torch():
    """All 2^32 binary32 inputs: oracle RN16 == torch's float16 cast (NaN -> some NaN)."""
    _exhaustive(to_bf16=False)


def test_bf16_converter_exhaustive_vs_torch():
    """All 2^32 binary32 inputs: oracle RNbf16 == torch's bfloat16 cast (NaN -> some NaN)."""
    _exhaustive(to_bf16=True)


def test_f16_converter_vs_numpy_sample():
    """A third opinion for FP16: numpy's own float16 cast on 2^22 random + edge patterns."""
    rng = np.random.default_rng(5)
    u = rng.integers(0, 1 << 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    edges = []
    for base in (0x33000000, 0x38800000, 0x477FE000, 0x477FF000, 0x3F801000, 0x00000001):
        edges.extend(range(max(0, base - 64), base + 64))
    u = np.concatenate([u, np.array(edges, dtype=np.uint32)])
    x = u.view(np.float32)
    x = x[np.isfinite(x)]
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.f32_to_f16_bits(x), ref)


def test_converters_exact_rounding_sample():
    """Rounding pinned to exact rational RNE on values near every rounding boundary."""
    rng = np.random.default_rng(11)
    u = rng.integers(0x00000001, 0x7F7FFFFF, size=3000, dtype=np.int64).astype(np.uint32)
    # force low mantissa bits to sit at/around the F16 and BF16 ties
    u[:1000] = (u[:1000] & ~np.uint32(0x1FFF)) | np.uint32(0x1000)
    u[1000:2000] = (u[1000:2000] & ~np.uint32(0xFFFF)) | np.uint32(0x8000)
    x = u.view(np.float32)
    x = np.concatenate([x, -x])
    h = oracle.f32_to_f16_bits(x)
    b = oracle.f32_to_bf16_bits(x)
    for xi, hi, bi in zip(x, h, b):
        v = exact.from_f32(xi)
        assert exact.output_bits(v, "f16") == int(hi), hex(int(np.array([xi]).view(np.uint32)[0]))
        assert exact.output_bits(v, "bf16") == int(bi), hex(int(np.array([xi]).view(np.uint32)[0]))


# ------------------------------------------------------- closed form grid
ENUM_OFFSETS = (1.0, -1.0, 1e-3, -1e-3, 0.0371, -0.0371, 0.52, -0.52)


@pytest.mark.parametrize("offset", ENUM_OFFSETS)
def test_every_scale_code_and_nibble_closed_form(offset):
    """Every (nested group, scale code, 4-bit code) against numpy float32 scalar ops."""
    p = gen.enumeration_problem(offset)
    nib = checker.unpack_nibbles(p.packed, p.n)
    outs = {o: oracle.dq4_nested(p, o) for o in OUTS}
    f32 = np.float32
    seen = set()
    for i in range(0, p.n):
        b = i // p.blocksize
        g = b // p.nested_blocksize
        key = (g, int(p.scale_codes[b]), int(nib[i]))
        if key in seen:
            continue
        seen.add(key)
        prod = f32(p.scale_codebook[key[1]]) * f32(p.nested_absmax[g])
        s = f32(prod) + f32(p.offset)
        v = f32(p.value_codebook[key[2]]) * f32(s)
        assert np.array([v]).view(np.uint32)[0] == outs["f32"][i:i + 1].view(np.uint32)[0]
        assert np.array([v]).astype(np.float16).view(np.uint16)[0] == outs["f16"][i]
        assert _torch_bits(np.array([v], dtype=np.float32), torch.bfloat16)[0] == outs["bf16"][i]
    assert len(seen) == 4 * 256 * 16


def test_fma_sentinel_is_covered():
    """The enumeration grid contains triples where a contracted multiply-add differs.

    For those the oracle must return the separately rounded scale; so an FMA
    anywhere (oracle or kernel) fails the closed-form and parity tests.
    """
    scb = gen.scale_codebook()
    total = 0
    for offset in ENUM_OFFSETS:
        p = gen.enumeration_problem(offset)
        hits = 0
        for g in range(p.ngroups):
            for k in range(256):
                sep = exact.nested_scale(scb[k], p.nested_absmax[g], offset)
                fma = exact.fma_scale(scb[k], p.nested_absmax[g], offset)
                if exact.f32_bits(sep) != exact.f32_bits(fma):
                    hits += 1
                    got = oracle.nested_scale(k, p.nested_absmax[g], scb, offset)
                    assert np.array([got]).view(np.uint32)[0] == exact.f32_bits(sep)
        assert hits > 0, offset
        total += hits
    assert total > 100


# ------------------------------------------------------------ brute force
def _random_problem(n, bs, nbs, fmt, offset, seed):
    return gen.make_problem(n, bs, nbs, fmt, 0.5, offset, seed)


def _brute_cases():
    cases = []
    for n in range(1, 301):
        cases.append((n, 32, 1))
    for n in range(1, 301, 7):
        cases.append((n, 64, 2))
        cases.append((n, 32, 256))
    for bs, nbs in ((32, 2), (64, 1), (32, 3)):
        for k in (1, 2, 3):
            for d in (-bs - 1, -bs + 1, -1, 0, 1, bs - 1, bs + 1):
                n = bs * nbs * k + d
                if n > 0:
                    cases.append((n, bs, nbs))
    return cases


def test_brute_force_tiny_against_exact_arithmetic():
    """Every value of ~700 tiny problems: oracle == exact rational evaluation, all dtypes.

    Covers partial outer blocks, partial nested groups (nested blocksizes 1, 2,
    3, 256) and both parities of n (odd n leaves a padding nibble).
    """
    for j, (n, bs, nbs) in enumerate(_brute_cases()):
        fmt = "nf4" if j % 2 else "fp4"
        offset = (0.52, -0.52, 1e-3, -1.0)[j % 4]
        p = _random_problem(n, bs, nbs, fmt, offset, 1000 + j)
        ex = exact.dequantize(p)
        for out in OUTS:
            got = _bits(oracle.dq4_nested(p, out), out)
            assert got == ex[out], (n, bs, nbs, out)


# --------------------------------------------------------- special cases
def test_identity_scale_reduces_to_codebook():
    """offset 0 and nested absmax 1: scale == scale_codebook[code] exactly; vcb = +-1 gives +-scale."""
    scb = gen.scale_codebook()
    for k in range(256):
        s = oracle.nested_scale(k, 1.0, scb, 0.0)
        assert np.array([s]).view(np.uint32)[0] == np.array([scb[k]]).view(np.uint32)[0]
    n = 256 * 32
    vcb = np.zeros(16, dtype=np.float32)
    vcb[1], vcb[2] = 1.0, -1.0
    codes = np.arange(256, dtype=np.uint8)
    for nibble, sign in ((1, 1.0), (2, -1.0)):
        packed = np.full(n // 2, nibble * 17, dtype=np.uint8)
        p = gen.Problem(packed, codes, np.ones(1, np.float32), scb, vcb, np.float32(0.0), n, 32, 256)
        v = oracle.dq4_nested(p, "f32").reshape(256, 32)
        assert np.array_equal(v, np.repeat((sign * scb)[:, None], 32, axis=1))


def test_zero_codebook_entry_gives_signed_zero():
    scb = gen.scale_codebook()
    n = 256 * 32
    vcb = np.zeros(16, dtype=np.float32)
    vcb[5] = -0.0
    p = gen.Problem(np.full(n // 2, 0x55, np.uint8), np.arange(256, dtype=np.uint8),
                    np.array([1.5], np.float32), scb, vcb, np.float32(0.25), n, 32, 256)
    v = oracle.dq4_nested(p, "f32").reshape(256, 32)
    s = scb.astype(np.float32) * np.float32(1.5) + np.float32(0.25)
    assert np.all(v == 0)
    assert np.array_equal(np.signbit(v), np.repeat((~np.signbit(s))[:, None], 32, axis=1))


def test_fused_equals_unfused_sequence_on_cpu():
    """Steps 1-2 (FP32 scale buffer) followed by the plain dequant == the fused definition."""
    for name in ("C2a", "C2b"):
        cell = gen.CELLS[name]
        p = cell.problem()
        s = oracle.nested_scales(p)
        assert np.array_equal(oracle.dq4(p.packed, s, p.value_codebook, p.n, p.blocksize, cell.out)
                              .view(np.uint8), oracle.dq4_nested(p, cell.out).view(np.uint8))


# ------------------------------------------- second implementation (numpy)
def _check_cell(p, out):
    a = oracle.dq4_nested(p, out, threads=8)
    b = checker.dq4_nested(p, out)
    assert a.view(np.uint8).tobytes() == b.view(np.uint8).tobytes()


@pytest.mark.parametrize("name", ["C1", "C2a", "C2b", "C3a", "C3d", "C5-bs32-off-0.001",
                                  "C5-bs4096-off+1"])
def test_numpy_checker_equals_oracle_on_cells(name):
    cell = gen.CELLS[name]
    _check_cell(cell.problem(), cell.out)


def test_numpy_checker_equals_oracle_on_tail_suite():
    for name, p, out in gen.tail_suite():
        _check_cell(p, out)


def test_threaded_oracle_equals_single_thread():
    p = gen.CELLS["C2a"].problem()
    assert np.array_equal(oracle.dq4_nested(p, "bf16", threads=1),
                          oracle.dq4_nested(p, "bf16", threads=5))


def test_transposed_oracle_index_map():
    """W^T output: out[c*rows + r] is the value (r, c) of the flat row-major definition.

    Pinned against numpy's transpose of the flat oracle (itself pinned above)
    and against exact evaluation of single elements.
    """
    for rows, cols, bs, nbs in ((1, 1, 32, 1), (3, 5, 32, 1), (65, 130, 32, 2), (64, 64, 64, 256),
                                (17, 4096, 4096, 1), (4097, 3, 64, 256)):
        p = gen.make_problem(rows * cols, bs, nbs, "fp4", 0.5, -0.52, seed=rows * 7 + cols)
        ex = exact.dequantize(p) if rows * cols <= 5000 else None
        for out in OUTS:
            t = oracle.dq4_nested_transposed(p, rows, cols, out)
            flat = oracle.dq4_nested(p, out)
            assert np.array_equal(t.reshape(cols, rows).view(np.uint8),
                                  np.ascontiguousarray(flat.reshape(rows, cols).T).view(np.uint8))
            if ex is not None:
                for r, c in ((0, 0), (rows - 1, cols - 1), (rows // 2, cols // 3)):
                    got = _bits(t[c * rows + r:c * rows + r + 1], out)[0]
                    assert got == ex[out][r * cols + c], (rows, cols, r, c, out)
