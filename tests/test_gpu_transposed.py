"""Transposed-output dequantization on the GPU, bit for bit against the oracle.

dq4_nested_transposed writes W^T for the row-major rows x cols weight W:
out[c * rows + r] is value (r, c) ("Fuse nested scale reconstruction into
SM103 4-bit dequantization", bitsandbytes issue #21, section "Correctness
requirements": transposed output must stay bitwise identical).
"""

import numpy as np
import pytest
import torch

import dq4_inputs as gen
import oracle

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
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


def bits(t):
    t = t.detach().reshape(-1).cpu()
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16).numpy().view(
        np.uint32 if t.dtype == torch.float32 else np.uint16)


def want_bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


def run(dq, p, t, rows, cols, kind, **kw):
    return dq.dq4_nested_transposed(t["packed"], t["scale_codes"], t["nested_absmax"],
                                    t["scale_codebook"], t["value_codebook"], float(p.offset),
                                    rows, cols, p.blocksize, p.nested_blocksize, DT[kind], **kw)


def check(dq, p, rows, cols, kind, threads=16, **kw):
    t = to_dev(p)
    got = run(dq, p, t, rows, cols, kind, **kw)
    want = oracle.dq4_nested_transposed(p, rows, cols, kind, threads=threads)
    g, w = bits(got), want_bits(want)
    if not np.array_equal(g, w):
        bad = np.flatnonzero(g != w)
        raise AssertionError(f"{rows}x{cols} {kind}: {bad.size} values differ, first {bad[:5]}")


SHAPES = [
    (1, 1), (1, 8), (8, 1), (3, 5), (63, 65), (64, 64), (65, 64), (64, 72), (127, 129),
    (96, 40), (200, 8), (8, 200), (1, 4096), (4096, 1), (130, 1000), (1000, 130),
    (257, 264), (512, 4095), (4095, 512), (333, 777),
    # rows % 4 == 0 and cols % 32 == 0 with partial row tiles: 16-bit outputs take the
    # 8-byte (four-row) stores there
    (100, 96), (260, 320), (4, 32), (132, 4096),
    # the staged kernel (cols % 32 == 0): partial 128-row and 256-column CTA tiles, a last
    # warp tile of 32 columns, one warp tile, rows % 8 == 0 (16-bit four-row stores) and
    # rows % 4 == 0
    (8, 32), (64, 32), (72, 96), (136, 352), (1000, 160), (520, 4064), (16, 8192),
    (12, 64),
]


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_small_shapes_all_dtypes(dq, rows, cols):
    for bs, nbs in ((32, 1), (64, 256), (4096, 2)):
        p = gen.make_problem(rows * cols, bs, nbs, "nf4" if bs == 64 else "fp4", 0.5, -0.52,
                             seed=rows * 1000 + cols + bs)
        for kind in DT:
            check(dq, p, rows, cols, kind, threads=1)


@pytest.mark.parametrize("name,rows,cols", [("C3a", 11008, 4096), ("C3c", 4096, 11008),
                                            ("C2a", 4097, 4095), ("C2b", 4097, 4095),
                                            ("C1", 4096, 4096)])
def test_cells(dq, name, rows, cols):
    cell = gen.CELLS[name]
    check(dq, cell.problem(), rows, cols, cell.out)


@pytest.mark.parametrize("kind", ["bf16", "f16"])
def test_grid_of_one_to_one_and_a_half_waves(dq, kind):
    """A grid of more than one and at most 1.5 waves of 8 CTAs per SM (the four-row kernel
    then runs its 6-CTA-per-SM build), with a partial last row tile and column tile."""
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    rows = 4100  # 33 row tiles, the last of 4 rows
    ct = -(-int(8 * sms * 1.06) // 33)
    cols = 256 * ct - 96  # ct column tiles, the last of 160 columns
    tiles = 33 * ct
    assert 8 * sms < tiles and 2 * tiles <= 3 * 8 * sms
    p = gen.make_problem(rows * cols, 64, 256, "nf4", 1.0, 0.1, seed=cols + len(kind))
    check(dq, p, rows, cols, kind)


@pytest.mark.parametrize("name", ["C4a", "C4d"])
def test_large_weight(dq, name):
    cell = gen.CELLS[name]
    check(dq, cell.problem(), cell.rows, cell.cols, cell.out)


@pytest.mark.parametrize("rows,cols", [(65540, 32800), (65537, 32771)])
def test_beyond_2_pow_31_values(dq, rows, cols):
    """rows x cols > 2^31 values (64-bit value and output indices), on the staged kernel
    (cols % 32 == 0; partial last row and column tiles) and on the odd-shape one (odd n):
    whole rows of W, read back from W^T, against the oracle on windows of whole nested
    groups: the first rows, the rows across flat index 2^31, and the last rows."""
    n = rows * cols
    assert n > (1 << 31)
    p = gen.make_problem(n, 64, 256, "nf4", 0.5, 0.0371, seed=rows + cols)
    t = to_dev(p)
    out = run(dq, p, t, rows, cols, "f16")
    torch.cuda.synchronize()
    wt = out.view(cols, rows)
    unit = 64 * 256
    r_mid = (1 << 31) // cols
    for r0 in (0, r_mid - 1, rows - 3):
        r1 = min(rows, r0 + 3)
        lo = (r0 * cols) // unit * unit
        hi = min(n, -(-(r1 * cols) // unit) * unit)
        sub = gen.Problem(p.packed[lo // 2:(hi + 1) // 2], p.scale_codes[lo // 64:-(-hi // 64)],
                          p.nested_absmax[lo // unit:-(-hi // unit)], p.scale_codebook,
                          p.value_codebook, p.offset, hi - lo, 64, 256)
        want = oracle.dq4_nested(sub, "f16")[r0 * cols - lo:r1 * cols - lo]
        got = wt[:, r0:r1].t().contiguous()
        assert np.array_equal(bits(got), want_bits(want)), (rows, cols, r0)
    del out, wt, t
    torch.cuda.empty_cache()


def test_every_code_transposed(dq):
    p = gen.enumeration_problem(0.52, blocksize=32, groups=4)
    rows, cols = 256, p.n // 256
    for kind in DT:
        check(dq, p, rows, cols, kind, threads=1)


def test_unaligned_output_and_canaries(dq):
    rows, cols = 200, 136
    p = gen.make_problem(rows * cols, 64, 256, "fp4", 0.5, 0.1, seed=5)
    t = to_dev(p)
    for kind in DT:
        isz = torch.empty(0, dtype=DT[kind]).element_size()
        guard = 4096
        buf = torch.full((rows * cols * isz + 2 * guard + isz,), 0x5A, dtype=torch.uint8,
                         device=DEV)
        # out shifted by one element: 16-byte stores cannot be used
        view = buf[guard + isz:guard + isz + rows * cols * isz].view(DT[kind])
        run(dq, p, t, rows, cols, kind, out=view)
        host = buf.cpu().numpy()
        assert np.all(host[:guard + isz] == 0x5A) and np.all(host[guard + isz + rows * cols * isz:]
                                                             == 0x5A), kind
        assert np.array_equal(bits(view), want_bits(oracle.dq4_nested_transposed(p, rows, cols,
                                                                                  kind)))


@pytest.mark.parametrize("shift", [1, 2, 4, 8])
def test_packed_off_sixteen_byte_boundaries(dq, shift):
    """`packed` 1, 2, 4 or 8 bytes past a 16-byte boundary: the odd-shape kernel takes every
    shape then (cols % 32 == 0 too), staging whole words when `packed` is 4-byte aligned and
    single bytes otherwise; W^T stays bit-exact."""
    for rows, cols in ((200, 160), (333, 777), (130, 96), (64, 4101)):
        p = gen.make_problem(rows * cols, 64, 256, "nf4", 0.5, 0.0371, seed=rows + cols + shift)
        t = to_dev(p)
        buf = torch.zeros(t["packed"].numel() + 16, dtype=torch.uint8, device=DEV)
        base = (16 - buf.data_ptr() % 16) % 16
        view = buf[base + shift:base + shift + t["packed"].numel()]
        view.copy_(t["packed"])
        assert view.data_ptr() % 16 == shift
        t2 = dict(t, packed=view)
        for kind in DT:
            got = dq.dq4_nested_transposed(t2["packed"], t2["scale_codes"], t2["nested_absmax"],
                                           t2["scale_codebook"], t2["value_codebook"],
                                           float(p.offset), rows, cols, p.blocksize,
                                           p.nested_blocksize, DT[kind])
            want = oracle.dq4_nested_transposed(p, rows, cols, kind, threads=1)
            assert np.array_equal(bits(got), want_bits(want)), (rows, cols, kind, shift)


def test_staged_path_stays_inside_out(dq):
    """Ragged shapes on the staged kernel (rows and cols not multiples of its tiles, out
    16-byte aligned inside a guarded buffer): W^T is written exactly and nothing around
    it."""
    for rows, cols in ((200, 160), (72, 96), (8, 32)):
        p = gen.make_problem(rows * cols, 32, 256, "nf4", 0.5, -0.0371, seed=rows + cols)
        t = to_dev(p)
        for kind in DT:
            isz = torch.empty(0, dtype=DT[kind]).element_size()
            guard = 4096
            buf = torch.full((rows * cols * isz + 2 * guard,), 0x5A, dtype=torch.uint8,
                             device=DEV)
            view = buf[guard:guard + rows * cols * isz].view(DT[kind])
            run(dq, p, t, rows, cols, kind, out=view)
            host = buf.cpu().numpy()
            assert np.all(host[:guard] == 0x5A) and np.all(host[guard + rows * cols * isz:]
                                                           == 0x5A), (rows, cols, kind)
            assert np.array_equal(bits(view), want_bits(
                oracle.dq4_nested_transposed(p, rows, cols, kind))), (rows, cols, kind)


def test_zero_and_errors(dq):
    p = gen.make_problem(64, 64, 256, "nf4", 0.5, 0.1, seed=1)
    t = to_dev(p)
    z = run(dq, p, t, 0, 17, "f16")
    assert z.numel() == 0
    with pytest.raises(dq.Dq4Error, match="BLOCKSIZE"):
        dq.dq4_nested_transposed(t["packed"], t["scale_codes"], t["nested_absmax"],
                                 t["scale_codebook"], t["value_codebook"], 0.1, 8, 8, 8192, 256)
