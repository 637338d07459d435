"""Pin of the row-blocked out_prod oracle (no GPU): on an integer-valued problem
W^T G equals sums of Python integers, entry by entry ("cuda: out_prod
dequantizes a 2D weight in row blocks", llama.cpp pull request #4, section
"What": out_prod sums over the weight's rows)."""

import numpy as np

import dq4_inputs as gen
import oracle
from tests import exact


def test_integer_problem_values_are_exact_integers():
    p = gen.make_integer_problem(300, 64, seed=3)
    ex = exact.dequantize(p, outs=("f32",))["f32"]
    w = np.array(ex, dtype=np.uint32).view(np.float32).reshape(300, 64)
    assert np.all(w == np.round(w)) and np.abs(w).max() <= 16
    assert np.array_equal(w, oracle.dq4_nested(p, "f32").reshape(300, 64))


def test_out_prod_matches_integer_sums():
    rows, cols, ncols = 257, 96, 5
    p = gen.make_integer_problem(rows, cols, seed=4)
    G = gen.make_ternary_g(rows, ncols, seed=5)
    d = oracle.out_prod(p, rows, cols, G)
    w = oracle.dq4_nested(p, "f32").reshape(rows, cols)
    wi = [[int(x) for x in row] for row in w]
    gi = [[int(x) for x in row] for row in G]
    for c in (0, 17, cols - 1):
        for j in range(ncols):
            assert d[c, j] == sum(wi[r][c] * gi[r][j] for r in range(rows))
