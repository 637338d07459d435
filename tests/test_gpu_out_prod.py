"""Row-blocked dequantization fused into a tcgen05 GEMM (dst = W^T G), on the GPU.

"cuda: out_prod dequantizes a 2D weight in row blocks" (llama.cpp pull
request #4): the weight's row blocks are dequantized to FP32 and a GEMM
accumulates them into dst, so the whole dequantized weight never exists; its
three new cases run k = 600000 rows at m = 256.  Here the row blocks are
decoded inside the GEMM kernel and the FP32 products come from three BF16
terms per operand.  Checks: (1) the decoded weight bit for bit: a G with one
1 per column makes each column of dst one row of W, exactly ("Fuse nested
scale reconstruction into SM103 4-bit dequantization", section "Correctness
requirements": the dequantized tensor passes bitwise equality before any GEMM
tolerance); (2) integer-valued problems, where every partial sum is an exact
integer below 2^24, so dst must equal the float64 oracle exactly whatever the
summation order; (3) realistic NF4 data within an FP32 accumulation bound;
(4) determinism, the single-range and split paths, ragged tiles, errors.
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
    Gd = G if isinstance(G, torch.Tensor) else torch.from_numpy(G).to(DEV)
    return dq.out_prod(t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
                       t["value_codebook"], float(p.offset), rows, cols, Gd, p.blocksize,
                       p.nested_blocksize, **kw)


NONE = torch.empty(0, dtype=torch.float32, device=DEV) if torch.cuda.is_available() else None


# (rows, cols, ncols, workspace): "auto" = the cached workspace (row ranges over the SMs),
# "none" = one range straight into dst, an int = a workspace of that many bytes
@pytest.mark.parametrize("rows,cols,ncols,ws", [
    (600000, 256, 64, "auto"),    # the page's row count: 76 ranges of 124 stages
    (600000, 256, 64, "none"),    # one range per CTA: 9375 stages each
    (5000, 100, 7, "auto"),       # a partial W-column tile, a 16-wide G tile, 4-byte G rows
    (4097, 4095, 3, "auto"),      # odd columns: 32 W-column tiles, rows not byte-aligned
    (1, 64, 1, "auto"),           # one row: a partial stage
    (3000, 512, 300, "auto"),     # three G tiles of 128, the last ragged
    (70000, 128, 256, 2 * 128 * 256 * 4),  # two G tiles, a workspace for two ranges only
])
def test_integer_exact(dq, rows, cols, ncols, ws):
    p = gen.make_integer_problem(rows, cols, seed=rows % 97)
    G = gen.make_ternary_g(rows, ncols, seed=cols)
    kw = {}
    if ws == "none":
        kw["workspace"] = NONE
    elif isinstance(ws, int):
        kw["workspace"] = torch.empty(ws // 4, dtype=torch.float32, device=DEV)
    bad = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = run(dq, p, rows, cols, G, bad=bad, **kw).cpu().numpy()
    want = oracle.out_prod(p, rows, cols, G, threads=16)
    assert np.array_equal(got.astype(np.float64), want), np.abs(got - want).max()
    assert int(bad.item()) == 0


@pytest.mark.parametrize("fmt,bs,nbs,offset,rows,cols", [
    ("nf4", 64, 256, 0.0371, 2048, 384),
    ("fp4", 32, 256, -0.52, 1536, 256),
    ("nf4", 4096, 256, 0.52, 1024, 1000),   # blocks span rows; a ragged W-column tile
    ("fp4", 128, 1, -0.0371, 777, 130),     # nested blocksize 1, odd rows, ragged tiles
])
def test_decoded_rows_bit_exact(dq, fmt, bs, nbs, offset, rows, cols):
    """G with one 1 per column: column j of dst is row r_j of W, bit for bit (both zeros
    compare equal: a GEMM adds +0 and -0 terms); every row of W is visited."""
    p = gen.make_problem(rows * cols, bs, nbs, fmt, 0.5, offset, seed=rows + bs)
    w = oracle.dq4_nested(p, "f32", threads=16).reshape(rows, cols)
    t = to_dev(p)
    ncols = 256
    order = np.argsort(gen.splitmix64(rows, 91, rows), kind="stable")
    for j0 in range(0, rows, ncols):
        sel = order[j0:j0 + ncols]
        G = torch.zeros((rows, ncols), dtype=torch.float32, device=DEV)
        G[torch.from_numpy(sel).to(DEV), torch.arange(sel.size, device=DEV)] = 1.0
        got = dq.out_prod(t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
                          t["value_codebook"], float(p.offset), rows, cols, G, bs,
                          nbs).cpu().numpy()[:, :sel.size]
        want = w[sel].T
        same = (got.view(np.uint32) == want.view(np.uint32)) | ((got == 0) & (want == 0))
        assert same.all(), (j0, int((~same).sum()))


def test_decoded_rows_bit_exact_beyond_2_pow_31_values(dq):
    """rows x cols > 2^31 weight values (64-bit value indices): G picks 16 rows of W (the
    first, the last, the two at flat index 2^31 and 12 others), and each column of dst must
    be its row of W bit for bit, against the oracle on windows of whole nested groups."""
    rows, cols, bs, nbs = (1 << 23) + 64, 256, 64, 256
    n = rows * cols
    assert n > (1 << 31)
    p = gen.make_problem(n, bs, nbs, "nf4", 0.5, 0.0371, seed=rows % 1009)
    t = to_dev(p)
    mid = (1 << 31) // cols  # the first row at flat index >= 2^31
    perm = np.argsort(gen.splitmix64(rows, 93, rows), kind="stable")
    picks = [0, rows - 1, mid - 1, mid]
    sel = np.array(picks + [int(r) for r in perm if int(r) not in picks][:12], dtype=np.int64)
    ncols = sel.size
    G = torch.zeros((rows, ncols), dtype=torch.float32, device=DEV)
    G[torch.from_numpy(sel).to(DEV), torch.arange(ncols, device=DEV)] = 1.0
    got = dq.out_prod(t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
                      t["value_codebook"], float(p.offset), rows, cols, G, bs, nbs).cpu().numpy()
    unit = bs * nbs
    for j, r in enumerate(sel):
        lo = (int(r) * cols) // unit * unit
        hi = min(n, lo + unit)
        sub = gen.Problem(p.packed[lo // 2:hi // 2], p.scale_codes[lo // bs:-(-hi // bs)],
                          p.nested_absmax[lo // unit:-(-hi // unit)], p.scale_codebook,
                          p.value_codebook, p.offset, hi - lo, bs, nbs)
        want = oracle.dq4_nested(sub, "f32")[int(r) * cols - lo:(int(r) + 1) * cols - lo]
        col = np.ascontiguousarray(got[:, j])
        same = (col.view(np.uint32) == want.view(np.uint32)) | ((col == 0) & (want == 0))
        assert same.all(), (int(r), int((~same).sum()))
    del t, G
    torch.cuda.empty_cache()


def test_realistic_weights_within_fp32_accumulation_tolerance(dq):
    rows, cols, ncols = 200000, 256, 32
    p = gen.make_problem(rows * cols, 64, 256, "nf4", 1.0, -0.1, seed=13)
    G = gen.make_normal_g(rows, ncols, seed=14)
    got = run(dq, p, rows, cols, G).cpu().numpy().astype(np.float64)
    want = oracle.out_prod(p, rows, cols, G, threads=16)
    w = oracle.dq4_nested(p, "f32", threads=16).reshape(rows, cols).astype(np.float64)
    # FP32 accumulation: |err| <= 4 u K^(3/2) rms(w g) per entry (u = 2^-24), far below a
    # missing or doubled block, which would shift an entry by ~sqrt(K / nblocks) rms(w g)
    rms = np.sqrt((w * w).T @ (G.astype(np.float64) ** 2) / rows)
    tol = 4 * 2.0 ** -24 * rows ** 1.5 * rms + 1e-30
    err = np.abs(got - want)
    assert np.all(err <= tol), float((err / tol).max())
    assert float((err / tol).max()) < 0.5
    # the three-term products: every entry within 8 u K rms(w g) (measured: 2.7).  The tensor
    # pipe's FP32 accumulation loses up to about an ulp of the accumulator per MMA, six MMAs
    # per K step here, so the error grows with the accumulation length like u K, not u
    # sqrt(K); a single BF16 term per operand would be off by ~2^-8 sqrt(K) rms, about 280
    # u K rms at K = 200000
    assert float((err / (2.0 ** -24 * rows * rms)).max()) < 8.0


def test_split_and_single_range_agree_and_repeat(dq):
    rows, cols, ncols = 50000, 256, 128
    p = gen.make_problem(rows * cols, 64, 256, "nf4", 0.5, 0.0371, seed=15)
    G = torch.from_numpy(gen.make_normal_g(rows, ncols, seed=16)).to(DEV)
    split = [run(dq, p, rows, cols, G) for _ in range(3)]
    one = run(dq, p, rows, cols, G, workspace=NONE)
    torch.cuda.synchronize()
    assert torch.equal(split[0], split[1]) and torch.equal(split[0], split[2])
    want = oracle.out_prod(p, rows, cols, G.cpu().numpy(), threads=16)
    scale = np.abs(want).max()
    # both within 2e-5 of the largest entry: the kernel adds its accumulator into the output
    # in FP32 every 512 rows, so one range over all 50000 rows is as accurate as many
    for got in (split[0], one):
        assert np.abs(got.cpu().numpy() - want).max() <= 2e-5 * scale


@pytest.mark.parametrize("rows,cols,ncols", [(20000, 256, 64), (3000, 512, 300), (777, 384, 16),
                                             (10, 256, 8), (63, 512, 100)])
def test_tma_and_copy_staging_agree(dq, rows, cols, ncols):
    """The same problem through the TMA staging (G 16-byte aligned) and the cp.async staging
    (G one float off 16 bytes): the decode and the MMA order are the same, so dst agrees bit
    for bit, and both are exact on integer-valued data."""
    p = gen.make_integer_problem(rows, cols, seed=rows % 89)
    G = torch.from_numpy(gen.make_ternary_g(rows, ncols, seed=cols)).to(DEV)
    buf = torch.empty(rows * ncols + 4, dtype=torch.float32, device=DEV)
    G1 = buf[1:1 + rows * ncols].view(rows, ncols)  # 4 bytes past a 16-byte boundary
    G1.copy_(G)
    assert G.data_ptr() % 16 == 0 and G1.data_ptr() % 16 == 4
    a = run(dq, p, rows, cols, G).cpu()
    b = run(dq, p, rows, cols, G1).cpu()
    assert torch.equal(a, b)
    want = oracle.out_prod(p, rows, cols, G.cpu().numpy(), threads=16)
    assert np.array_equal(a.numpy().astype(np.float64), want)


def test_zero_rows_and_errors(dq):
    p = gen.make_integer_problem(64, 64, seed=1)
    t = to_dev(p)
    G = torch.zeros((0, 3), dtype=torch.float32, device=DEV)
    dst = torch.full((64, 3), 5.0, device=DEV)
    dq.out_prod(t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
                t["value_codebook"], 0.0, 0, 64, G, dst=dst)
    assert torch.count_nonzero(dst).item() == 0
    G2 = torch.zeros((64, 3), dtype=torch.float32, device=DEV)
    buf = torch.zeros(16, dtype=torch.float32, device=DEV)
    st = dq.lib.dq4_nested_out_prod(
        t["packed"].data_ptr(), t["scale_codes"].data_ptr(), t["nested_absmax"].data_ptr(),
        t["scale_codebook"].data_ptr(), t["value_codebook"].data_ptr(), 0.0, 64, 64, 64, 256,
        G2.data_ptr(), 3, dst.data_ptr(), buf.data_ptr() + 2, 32, None, None)
    assert st == 6  # DQ4_ERR_ALIGN: a workspace that is not 4-byte aligned
    with pytest.raises(ValueError, match="rows x ncols"):
        dq.out_prod(t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
                    t["value_codebook"], 0.0, 64, 64, G2[:10])
