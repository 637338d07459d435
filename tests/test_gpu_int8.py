"""LLM.int8 correction-operand preparation on the GPU, bit for bit against the oracle.

"Fuse LLM.int8 correction operand preparation into one CUDA kernel"
(bitsandbytes issue #16), section "Exact correctness oracle": raw-bit equality
for subA and for the FP16 subB, over the preparation grid of section "B300
benchmark plan" (M x K/N x L), first/last/noncontiguous/sorted/repeated
columns, and the empty-outlier case.
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


def dev_inputs(p, dtype=torch.float16):
    A = torch.from_numpy(p.A_bits).to(DEV).view(dtype)
    CB = torch.from_numpy(p.CB).to(DEV)
    SCB = torch.from_numpy(p.SCB).to(DEV)
    cols = torch.from_numpy(p.cols).to(DEV)
    return A, CB, SCB, cols


def bits16(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def check(dq, p, dtype=torch.float16):
    A, CB, SCB, cols = dev_inputs(p, dtype)
    subA, subB = dq.int8_correction_prep(A, CB, SCB, cols)
    wa, wb = oracle.int8_correction_prep(p.A_bits, p.CB, p.SCB, p.cols)
    assert np.array_equal(bits16(subA), wa), p.shape
    gb = bits16(subB)
    if not np.array_equal(gb, wb):
        bad = np.argwhere(gb != wb)
        raise AssertionError(f"{p.shape}: {len(bad)} subB values differ, first {bad[:3]}")


@pytest.mark.parametrize("KN", gen.INT8_GRID_KN)
@pytest.mark.parametrize("M", gen.INT8_GRID_M)
def test_preparation_grid(dq, M, KN):
    """Every L of the grid, plus the ~1% control, on one (M, K = N) pair."""
    base = gen.make_int8_problem(M, KN, KN, 64, seed=M + KN)
    for L in gen.INT8_GRID_L + (KN // 100,):
        sub = gen.make_int8_problem(1, 1, KN, L, seed=M * 3 + L)  # columns only
        p = gen.Int8Problem(base.A_bits, base.CB, base.SCB, sub.cols)
        check(dq, p)


@pytest.mark.parametrize("mode", ["sorted", "unsorted", "repeated", "edges"])
def test_column_modes(dq, mode):
    check(dq, gen.make_int8_problem(64, 4096, 4096, 64, seed=9, cols_mode=mode))


def test_rectangular_odd_and_bf16(dq):
    check(dq, gen.make_int8_problem(33, 1001, 777, 17, seed=4, cols_mode="unsorted"))  # odd N
    check(dq, gen.make_int8_problem(5, 3, 3584, 5, seed=6, cols_mode="edges"))
    check(dq, gen.make_int8_problem(64, 4096, 8192, 16, seed=7), dtype=torch.bfloat16)
    check(dq, gen.make_int8_problem(0, 512, 256, 8, seed=8))    # no activations
    check(dq, gen.make_int8_problem(16, 0, 256, 8, seed=9))     # no weights


def test_empty_outliers_is_a_no_op(dq):
    p = gen.make_int8_problem(8, 64, 64, 0, seed=1)
    A, CB, SCB, cols = dev_inputs(p)
    subA = torch.full((8, 0), 7, dtype=torch.float16, device=DEV)
    subB = torch.empty((0, 64), dtype=torch.float16, device=DEV)
    a, b = dq.int8_correction_prep(A, CB, SCB, cols, subA=subA, subB=subB)
    assert a.numel() == 0 and b.numel() == 0


def test_out_of_range_columns_are_counted_and_zeroed(dq):
    p = gen.make_int8_problem(4, 96, 100, 6, seed=2, cols_mode="unsorted")
    good = p.cols.copy()
    cols = good.copy()
    cols[1], cols[4] = -3, 100  # two invalid entries
    A, CB, SCB, _ = dev_inputs(p)
    bad = torch.zeros(1, dtype=torch.int32, device=DEV)
    subA, subB = dq.int8_correction_prep(A, CB, SCB, torch.from_numpy(cols).to(DEV),
                                         bad_cols=bad)
    torch.cuda.synchronize()
    assert int(bad.item()) == 2
    wa, wb = oracle.int8_correction_prep(p.A_bits, p.CB, p.SCB, good)
    ga, gb = bits16(subA), bits16(subB)
    keep = [0, 2, 3, 5]
    assert np.array_equal(ga[:, keep], wa[:, keep]) and np.all(ga[:, [1, 4]] == 0)
    assert np.array_equal(gb[keep], wb[keep]) and np.all(gb[[1, 4]] == 0)


def test_unaligned_subB_and_repeated_calls(dq):
    p = gen.make_int8_problem(8, 512, 4096, 16, seed=12)
    A, CB, SCB, cols = dev_inputs(p)
    buf = torch.empty(16 * 512 + 1, dtype=torch.float16, device=DEV)
    subB = buf[1:].view(16, 512)  # 2-byte aligned only: per-element stores
    for _ in range(2):
        subA, out = dq.int8_correction_prep(A, CB, SCB, cols, subB=subB)
    wa, wb = oracle.int8_correction_prep(p.A_bits, p.CB, p.SCB, p.cols)
    assert np.array_equal(bits16(out), wb) and np.array_equal(bits16(subA), wa)


def test_subA_several_elements_per_thread_ragged(dq):
    # M x L = 128961: more than three fills of the SMs, so each subA thread takes several
    # elements, and not a multiple of a CTA's share, so the last subA CTA is partial
    check(dq, gen.make_int8_problem(2047, 512, 4096, 63, seed=13, cols_mode="unsorted"))


def test_out_of_range_columns_counted_once_at_large_M(dq):
    p = gen.make_int8_problem(2047, 64, 4096, 63, seed=14, cols_mode="unsorted")
    good = p.cols.copy()
    cols = good.copy()
    cols[5], cols[40] = -1, 4096  # two invalid entries
    A, CB, SCB, _ = dev_inputs(p)
    bad = torch.zeros(1, dtype=torch.int32, device=DEV)
    subA, subB = dq.int8_correction_prep(A, CB, SCB, torch.from_numpy(cols).to(DEV),
                                         bad_cols=bad)
    torch.cuda.synchronize()
    assert int(bad.item()) == 2
    wa, wb = oracle.int8_correction_prep(p.A_bits, p.CB, p.SCB, good)
    ga, gb = bits16(subA), bits16(subB)
    keep = [l for l in range(63) if l not in (5, 40)]
    assert np.array_equal(ga[:, keep], wa[:, keep]) and np.all(ga[:, [5, 40]] == 0)
    assert np.array_equal(gb[keep], wb[keep]) and np.all(gb[[5, 40]] == 0)
