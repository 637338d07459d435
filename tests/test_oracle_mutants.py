"""The pins are strong enough: every planted mistake in the oracle fails one of them.

Each mutant is a copy of the C oracle with one plausible mistake (a dropped
term, a wrong sign, a wrong index, a transposed operand, a wrong rounding
rule, a contracted multiply-add), compiled into a temporary library on the
CPU.  The committed oracle itself is never modified.
"""

import os
import platform
import tempfile

import numpy as np
import pytest

import dq4_inputs as gen
import oracle
from tests import exact
from tests.test_oracle_pins import OUTS, _bits, _hand_problem, _load_cases

SRC = os.path.join(os.path.dirname(oracle.__file__), "dq4_oracle.c")

MUTANTS = {
    "nibble_order_swapped": ("(i % 2 == 0) ? (byte >> 4) : (byte & 0x0F)",
                             "(i % 2 == 0) ? (byte & 0x0F) : (byte >> 4)"),
    "offset_dropped": ("const float scale = product + offset;", "const float scale = product;"),
    "offset_sign_flipped": ("const float scale = product + offset;",
                            "const float scale = product - offset;"),
    "nested_group_index": ("const int64_t g = b / nested_blocksize;",
                           "const int64_t g = (b / nested_blocksize) / 2;"),
    "outer_block_index": ("const int64_t b = i / blocksize;",
                          "const int64_t b = i / (2 * blocksize);"),
    "codebook_operand_swapped": ("const float v = value_codebook[nibble_of(packed, i)] * scale;",
                                 "const float v = scale_codebook[nibble_of(packed, i)] * scale;"),
    "ties_away_from_zero": ("(rem == half && (R & 1ull))", "(rem == half)"),
    "truncation": ("if (rem > half || (rem == half && (R & 1ull))) R++;", "(void)half;"),
    "subnormals_flushed": ("int Q = (L > emin ? L : emin) - (p - 1);",
                           "int Q = L - (p - 1); if (L < emin) return sign;"),
    "no_overflow_to_inf": ("if (Q + (p - 1) > emax) return (uint16_t)(sign | exp_all_ones);",
                           "(void)emax;"),
}


def _fma_flags():
    extra = ["-ffp-contract=fast"]
    if platform.machine() in ("x86_64", "AMD64"):
        extra.append("-mfma")
    return extra


def _pins_pass(lib) -> bool:
    """A quick battery of the pins, run against the library ``lib``."""
    for case in _load_cases():
        p = _hand_problem(case)
        for out in OUTS:
            got = _bits(oracle.dq4_nested(p, out, lib=lib), out)
            want = ([int(h, 16) for h in case["expected_values"][out]]
                    if "expected_values" in case else [int(case["expected"][out], 16)] * p.n)
            if got != want:
                return False
    for j, (n, bs, nbs) in enumerate([(n, 32, 1) for n in range(1, 70)] +
                                     [(700, 32, 2), (2 * 32 * 3 + 5, 32, 3), (64 * 256 + 33, 64, 256)]):
        p = gen.make_problem(n, bs, nbs, "nf4" if j % 2 else "fp4", 0.5,
                             (0.52, -0.52, 1e-3, -1.0)[j % 4], 2000 + j)
        ex = exact.dequantize(p)
        for out in OUTS:
            if _bits(oracle.dq4_nested(p, out, lib=lib), out) != ex[out]:
                return False
    return True


def _compile(src_text: str, tmp: str, name: str, extra=None):
    path = os.path.join(tmp, f"{name}.c")
    with open(path, "w") as f:
        f.write(src_text)
    return oracle.load(oracle.build(force=True, src=path, dst=os.path.join(tmp, f"{name}.so"),
                                    extra_flags=extra))


def test_unmutated_copy_passes_battery():
    with tempfile.TemporaryDirectory() as tmp:
        with open(SRC) as f:
            lib = _compile(f.read(), tmp, "clean")
        assert _pins_pass(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) >= 1, f"mutation site for {name} not found"
    with tempfile.TemporaryDirectory() as tmp:
        lib = _compile(text.replace(old, new), tmp, name)
        assert not _pins_pass(lib), f"mutant {name} survived every pin"


def test_fma_contraction_is_caught():
    """Compiled with contraction allowed, the no-FMA golden case fails."""
    with open(SRC) as f:
        text = f.read()
    with tempfile.TemporaryDirectory() as tmp:
        lib = _compile(text, tmp, "fma", extra=_fma_flags())
        scb = np.array([np.uint32(0x3F7FFFFF)], dtype=np.uint32).view(np.float32)
        s = oracle.nested_scale(0, scb[0], scb, np.array([0xBF7FFFFE], np.uint32)
                                .view(np.float32)[0], lib=lib)
        if s == 0.0:
            pytest.skip("this compiler did not contract the multiply-add even when allowed")
        assert not _pins_pass(lib)
