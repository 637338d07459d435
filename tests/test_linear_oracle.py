"""Pins of the fused-linear oracle (no GPU).

The oracle's Y = X W^T is checked against facts outside it: the operand
bits come from the exact rational dequantization (``tests/exact.py``), the
16-bit decoding against patterns fixed by the formats, the orientation with
unit-vector activations, and the contraction against Python integer sums.
The path is the dequantize-plus-linear fallback of "Fuse nested scale
reconstruction into SM103 4-bit dequantization" (bitsandbytes issue #21,
section "Problem"): the weight expanded as dq4_nested does, then F.linear.
"""

import numpy as np
import pytest

import dq4_inputs as gen
import oracle
from tests import exact

ONE = {"bf16": 0x3F80, "f16": 0x3C00}
MINUS_ONE = {"bf16": 0xBF80, "f16": 0xBC00}


def weight_values(p, dtype, N, K):
    """W's values from the exact path: bits -> float64 by the formats' definitions."""
    bits = np.array(exact.dequantize(p, outs=(dtype,))[dtype], dtype=np.uint32)
    if dtype == "bf16":
        vals = (bits << 16).view(np.float32).astype(np.float64)
    else:
        vals = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    return vals.reshape(N, K)


def test_16bit_operand_decoding():
    bf = np.array([0x3F80, 0xC000, 0x0001, 0x7F7F, 0x8000], np.uint16)
    assert list(oracle._bits16_to_f64(bf, "bf16")) == [
        1.0, -2.0, 2.0 ** -133, (2 - 2.0 ** -7) * 2.0 ** 127, -0.0]
    h = np.array([0x3C00, 0xC000, 0x0001, 0x7BFF, 0x3555], np.uint16)
    assert list(oracle._bits16_to_f64(h, "f16")) == [
        1.0, -2.0, 2.0 ** -24, 65504.0, 1365.0 / 4096.0]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_unit_vectors_pick_weight_columns(dtype):
    """X row m = e_{k_m} gives Y[m, n] = W[n, k_m]: X W^T, not X W or W X^T."""
    N, K = 6, 96
    p = gen.make_integer_problem(N, K, blocksize=32, seed=11)
    ks = [0, 1, 31, 32, 63, 95, 17]
    X = np.zeros((len(ks), K), np.uint16)
    for m, k in enumerate(ks):
        X[m, k] = ONE[dtype]
    Y = oracle.linear(p, X, dtype, N, K, threads=2)
    W = weight_values(p, dtype, N, K)
    assert Y.shape == (len(ks), N)
    for m, k in enumerate(ks):
        assert np.array_equal(Y[m], W[:, k]), (m, k)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_matches_integer_sums(dtype):
    """Integer weights (|w| <= 16) and ternary activations: exact Python sums."""
    M, N, K = 5, 7, 128
    p = gen.make_integer_problem(N, K, blocksize=64, seed=12)
    G = gen.make_ternary_g(M, K, seed=13).astype(np.int64)
    X = np.where(G > 0, ONE[dtype], np.where(G < 0, MINUS_ONE[dtype], 0)).astype(np.uint16)
    Y = oracle.linear(p, X, dtype, N, K, threads=2)
    W = weight_values(p, dtype, N, K)
    wi = [[int(v) for v in row] for row in W]
    assert all(float(a) == b for row, rw in zip(wi, W) for a, b in zip(row, rw))
    for m in range(M):
        for n in range(N):
            s = sum(int(G[m, k]) * wi[n][k] for k in range(K))
            assert Y[m, n] == s, (m, n)


def test_linear_in_x():
    """Y(X1 + X2) = Y(X1) + Y(X2) for activations whose sum is exact in BF16."""
    N, K = 9, 64
    p = gen.make_integer_problem(N, K, seed=14)
    a = gen.make_ternary_g(3, K, seed=15)
    b = gen.make_ternary_g(3, K, seed=16)
    enc = {-2: 0xC000, -1: 0xBF80, 0: 0, 1: 0x3F80, 2: 0x4000}
    bits = lambda g: np.vectorize(enc.get)(g.astype(np.int64)).astype(np.uint16)
    ya, yb = (oracle.linear(p, bits(g), "bf16", N, K, threads=2) for g in (a, b))
    yab = oracle.linear(p, bits(a + b), "bf16", N, K, threads=2)
    assert np.array_equal(yab, ya + yb)
