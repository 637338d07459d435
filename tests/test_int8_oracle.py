"""Pins of the LLM.int8 correction-operand oracle (no GPU).

"Fuse LLM.int8 correction operand preparation into one CUDA kernel"
(bitsandbytes issue #16), section "Exact correctness oracle": raw-bit equality
for subA; raw-bit FP16 equality for subB with the order FP32 CB * SCB, then a
separately rounded FP32 multiplication by the reciprocal-127 constant, then
the FP16 conversion; the complete INT8 code domain; zero, normal,
subnormal-adjacent and large finite SCB; first, last, noncontiguous, sorted
and repeated columns.
"""

import os
import tempfile

import numpy as np
import pytest

import dq4_inputs as gen
import oracle
import oracle.checker as checker
from tests import exact

RECIP127 = np.float32(1) / np.float32(127)

SCB_SPECIAL = [0.0, 1e-45, 2.0 ** -149 * 3, 2.0 ** -126, 1.1754942e-38, 2.0 ** -100, 1e-3, 0.5,
               1.0, 3.7, 127.0, 1e4, 65504.0, 1e30, 3.4028235e38]


def _f16_bits_of_exact(v: exact.Val) -> int:
    return exact.output_bits(v, "f16")


def _expected_subB(code: int, scb: float) -> int:
    """RN16(RN32(RN32(code * scb) * RN32(1/127))) by exact arithmetic, infinities included."""
    t1 = exact.mul(exact.from_f32(code), exact.from_f32(scb))
    if t1.inf:
        return 0xFC00 if t1.neg else 0x7C00  # inf * (1/127) stays inf, which FP16 keeps
    t2 = exact.mul(t1, exact.from_f32(RECIP127))
    if t2.inf:
        return 0xFC00 if t2.neg else 0x7C00
    return _f16_bits_of_exact(t2)


def order_sensitive_cases(count: int = 64):
    """(code, scb) pairs where the other multiplication order changes the FP16 result.

    Found by a seeded search over lognormal SCB values with numpy float32
    arithmetic; every pair is then checked against exact arithmetic.
    """
    scb = gen.lognormal_f32(77, gen.STREAM_SCB, 1 << 16, 2.0)
    codes = np.arange(-128, 128, dtype=np.float32)
    c = np.repeat(codes, scb.size)
    sv = np.tile(scb, codes.size)
    with np.errstate(over="ignore"):
        right = ((c * sv) * RECIP127).astype(np.float16).view(np.uint16)
        other = ((c * RECIP127) * sv).astype(np.float16).view(np.uint16)
    idx = np.flatnonzero(right != other)[:count]
    return [(int(c[i]), float(sv[i])) for i in idx]


def test_order_sensitive_cases_exist_and_pass():
    cases = order_sensitive_cases()
    assert len(cases) >= 16
    cb = np.array([[c for c, _ in cases]], dtype=np.int8).T.copy()      # N x 1
    scb = np.array([s for _, s in cases], dtype=np.float32)
    _, subB = oracle.int8_correction_prep(np.zeros((1, 1), np.uint16), cb, scb,
                                          np.zeros(1, dtype=np.int64))
    for n, (c, sv) in enumerate(cases):
        assert int(subB[0, n]) == _expected_subB(c, sv), (c, sv)


def test_reciprocal_constant():
    assert np.array([RECIP127]).view(np.uint32)[0] == 0x3C010204
    # 127 * RN32(1/127) = 1 - 2^-28 exactly, which rounds to 1.0 in FP32
    assert exact.mul(exact.from_f32(127.0), exact.from_f32(RECIP127)).q == 1


def test_complete_int8_domain_and_special_scb():
    K = 256
    N = len(SCB_SPECIAL)
    cb = np.tile((np.arange(K) - 128).astype(np.int8), (N, 1))
    scb = np.array(SCB_SPECIAL, dtype=np.float32)
    cols = np.arange(K, dtype=np.int64)
    a = np.zeros((1, K), dtype=np.uint16)
    _, subB = oracle.int8_correction_prep(a, cb, scb, cols)
    for n in range(N):
        for k in range(K):
            assert int(subB[k, n]) == _expected_subB(k - 128, float(scb[n])), (k - 128, scb[n])


def test_hand_worked_cases():
    """CB = 127, SCB = 1: t1 = 127, t2 = 1 - 2^-28 rounds to 1.0 (FP16 0x3c00).
    CB = -1, SCB = 127: t1 = -127, t2 = -1.0 (0xbc00).  CB = 0: +0 or -0 by SCB sign is +0."""
    cb = np.array([[127, -1, 0]], dtype=np.int8).repeat(2, axis=0)
    scb = np.array([1.0, 127.0], dtype=np.float32)
    _, subB = oracle.int8_correction_prep(np.zeros((1, 3), np.uint16), cb, scb,
                                          np.arange(3, dtype=np.int64))
    assert subB[0, 0] == 0x3C00 and subB[1, 1] == 0xBC00 and subB[2, 0] == 0 and subB[2, 1] == 0


@pytest.mark.parametrize("mode", ["sorted", "unsorted", "repeated", "edges"])
def test_gather_semantics(mode):
    p = gen.make_int8_problem(7, 9, 300, 13, seed=3, cols_mode=mode)
    subA, subB = oracle.int8_correction_prep(p.A_bits, p.CB, p.SCB, p.cols)
    for m in range(7):
        for l in range(13):
            assert subA[m, l] == p.A_bits[m, p.cols[l]]
    for l in range(13):
        for n in range(9):
            assert int(subB[l, n]) == _expected_subB(int(p.CB[n, p.cols[l]]), float(p.SCB[n]))
    if mode == "edges":
        assert p.cols[0] == 0 and p.cols[-1] == 299
    if mode == "repeated":
        assert len(set(p.cols.tolist())) < p.cols.size


@pytest.mark.parametrize("M", [1, 64])
@pytest.mark.parametrize("KN", [3584, 4096])
@pytest.mark.parametrize("L", gen.INT8_GRID_L + (41,))
def test_checker_equals_oracle_on_grid(M, KN, L):
    p = gen.make_int8_problem(M, KN, KN, L, seed=M * 7 + L)
    a1, b1 = oracle.int8_correction_prep(p.A_bits, p.CB, p.SCB, p.cols)
    a2, b2 = checker.int8_correction_prep(p.A_bits, p.CB, p.SCB, p.cols)
    assert np.array_equal(a1, a2) and np.array_equal(b1, b2)


INT8_MUTANTS = {
    "recip_first": ("""            const float t1 = (float)CB[n * K + cols[l]] * SCB[n];   /* RN32(CB * SCB) */
            const float t2 = t1 * recip127;                         /* RN32(t1 * 1/127) */""",
                    """            const float t1 = (float)CB[n * K + cols[l]] * recip127;
            const float t2 = t1 * SCB[n];"""),
    "single_rounding": ("""            const float t2 = t1 * recip127;                         /* RN32(t1 * 1/127) */""",
                        """            const float t2 = (float)((double)CB[n * K + cols[l]] * SCB[n] / 127.0);
            (void)t1;"""),
    "untransposed": ("subB[l * N + n] = oracle_f32_to_f16(t2);",
                     "subB[n * L + l] = oracle_f32_to_f16(t2);"),
}


def _int8_pins_pass(lib) -> bool:
    K, N = 256, len(SCB_SPECIAL)
    cb = np.tile((np.arange(K) - 128).astype(np.int8), (N, 1))
    scb = np.array(SCB_SPECIAL, dtype=np.float32)
    _, subB = oracle.int8_correction_prep(np.zeros((1, K), np.uint16), cb, scb,
                                          np.arange(K, dtype=np.int64), lib=lib)
    for n in range(N):
        for k in range(K):
            if int(subB[k, n]) != _expected_subB(k - 128, float(scb[n])):
                return False
    cases = order_sensitive_cases()
    cbo = np.array([[c for c, _ in cases]], dtype=np.int8).T.copy()
    scbo = np.array([v for _, v in cases], dtype=np.float32)
    _, subBo = oracle.int8_correction_prep(np.zeros((1, 1), np.uint16), cbo, scbo,
                                           np.zeros(1, dtype=np.int64), lib=lib)
    for n, (c, v) in enumerate(cases):
        if int(subBo[0, n]) != _expected_subB(c, v):
            return False
    # a rectangular problem, element by element (shows a wrong layout)
    p = gen.make_int8_problem(3, 5, 40, 7, seed=1, cols_mode="unsorted")
    _, sb = oracle.int8_correction_prep(p.A_bits, p.CB, p.SCB, p.cols, lib=lib)
    for l in range(7):
        for n in range(5):
            if int(sb[l, n]) != _expected_subB(int(p.CB[n, p.cols[l]]), float(p.SCB[n])):
                return False
    return True


def test_int8_pins_pass_on_unmutated_copy():
    src = os.path.join(os.path.dirname(oracle.__file__), "dq4_oracle.c")
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "m.c")
        with open(path, "w") as f:
            f.write(open(src).read())
        assert _int8_pins_pass(oracle.load(oracle.build(force=True, src=path,
                                                        dst=os.path.join(tmp, "m.so"))))


@pytest.mark.parametrize("name", sorted(INT8_MUTANTS))
def test_int8_mutants_are_caught(name):
    old, new = INT8_MUTANTS[name]
    src = os.path.join(os.path.dirname(oracle.__file__), "dq4_oracle.c")
    text = open(src).read()
    assert old in text, name
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "m.c")
        with open(path, "w") as f:
            f.write(text.replace(old, new))
        lib = oracle.load(oracle.build(force=True, src=path, dst=os.path.join(tmp, "m.so")))
        assert not _int8_pins_pass(lib), f"mutant {name} survived"
