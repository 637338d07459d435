"""Row-blocked dequantization feeding cuBLAS GEMMs (dst = W^T G), on the GPU.

"cuda: out_prod dequantizes a 2D weight in row blocks" (llama.cpp pull
request #4): each row block is dequantized to FP32 into a bounded transient
and accumulated into dst by a GEMM with beta 0 for the first block and 1
after; its three new cases run k = 600000 rows at m = 256 (three blocks).
Checks: (1) integer-valued problems, where every FP32 partial sum is an exact
integer below 2^24, so dst must equal the float64 oracle exactly whatever
the GEMM's summation order; (2) the dequantized transient itself is
bit-identical to the oracle ("Fuse nested scale reconstruction into SM103
4-bit dequantization", section "Correctness requirements": the dequantized
tensor passes bitwise equality before any GEMM tolerance); (3) realistic
NF4 data with an FP32 accumulation tolerance.
"""

import numpy as np
import pytest
import torch

import dq4_inputs as gen
import oracle

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def dq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_weight_dequantization_gb300 as m
    return m


def to_dev(p):
    return {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(DEV)
            for k in ("packed", "scale_codes", "nested_absmax", "scale_codebook",
                      "value_codebook")}


def run(dq, p, rows, cols, G, **kw):
    t = to_dev(p)
    Gd = torch.from_numpy(G).to(DEV)
    return dq.out_prod(t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
                       t["value_codebook"], float(p.offset), rows, cols, Gd, p.blocksize,
                       p.nested_blocksize, **kw)


@pytest.mark.parametrize("rows,cols,ncols,budget", [
    (600000, 256, 64, 256 << 20),   # three blocks: 262144 + 262144 + 75712 rows
    (600000, 256, 64, 1 << 20),     # 1024-row blocks (586 of them)
    (5000, 100, 7, 100 * 4 * 37),   # 37-row blocks, not group-aligned: per-value path
    (4097, 4095, 3, 4095 * 4 * 1000),
    (1, 64, 1, 1 << 20),
])
def test_integer_exact(dq, rows, cols, ncols, budget):
    p = gen.make_integer_problem(rows, cols, seed=rows % 97)
    G = gen.make_ternary_g(rows, ncols, seed=cols)
    got = run(dq, p, rows, cols, G, transient_bytes=budget).cpu().numpy()
    want = oracle.out_prod(p, rows, cols, G, threads=16)
    assert np.array_equal(got.astype(np.float64), want), np.abs(got - want).max()


def test_transient_holds_the_last_block_bit_exact(dq):
    rows, cols, ncols = 3000, 512, 4
    p = gen.make_problem(rows * cols, 64, 256, "nf4", 0.5, 0.0371, seed=11)
    G = gen.make_normal_g(rows, ncols, seed=12)
    rb = 700  # a 700-row budget, aligned down to a multiple of 16384 / gcd(512, 16384) = 32
    transient = torch.empty(rb * cols, dtype=torch.float32, device=DEV)
    run(dq, p, rows, cols, G, transient=transient, transient_bytes=rb * cols * 4)
    torch.cuda.synchronize()
    blk = 672
    last0 = ((rows - 1) // blk) * blk
    w = oracle.dq4_nested(p, "f32").reshape(rows, cols)
    got = transient[:(rows - last0) * cols].cpu().numpy().reshape(rows - last0, cols)
    assert np.array_equal(got.view(np.uint32), w[last0:].view(np.uint32))


def test_realistic_weights_within_fp32_accumulation_tolerance(dq):
    rows, cols, ncols = 200000, 256, 32
    p = gen.make_problem(rows * cols, 64, 256, "nf4", 1.0, -0.1, seed=13)
    G = gen.make_normal_g(rows, ncols, seed=14)
    got = run(dq, p, rows, cols, G, transient_bytes=32 << 20).cpu().numpy().astype(np.float64)
    want = oracle.out_prod(p, rows, cols, G, threads=16)
    w = oracle.dq4_nested(p, "f32", threads=16).reshape(rows, cols).astype(np.float64)
    # FP32 accumulation: |err| <= 4 u K^(3/2) rms(w g) per entry (u = 2^-24), far below a
    # missing or doubled block, which would shift an entry by ~sqrt(K / nblocks) rms(w g)
    rms = np.sqrt((w * w).T @ (G.astype(np.float64) ** 2) / rows)
    tol = 4 * 2.0 ** -24 * rows ** 1.5 * rms + 1e-30
    err = np.abs(got - want)
    assert np.all(err <= tol), float((err / tol).max())
    assert float((err / tol).max()) < 0.5


def test_zero_rows_and_errors(dq):
    p = gen.make_integer_problem(64, 64, seed=1)
    t = to_dev(p)
    G = torch.zeros((0, 3), dtype=torch.float32, device=DEV)
    dst = torch.full((64, 3), 5.0, device=DEV)
    dq.out_prod(t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
                t["value_codebook"], 0.0, 0, 64, G, dst=dst)
    assert torch.count_nonzero(dst).item() == 0
    G2 = torch.zeros((64, 3), dtype=torch.float32, device=DEV)
    with pytest.raises(dq.Dq4Error, match="TOO_LARGE"):
        dq.out_prod(t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
                    t["value_codebook"], 0.0, 64, 64, G2,
                    transient=torch.empty(16, device=DEV), transient_bytes=64)
