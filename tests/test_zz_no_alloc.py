"""The allocation-free entry point dq4_nested_unfused_static, called through the C ABI.

Some callers cannot allocate device memory while they run: a serving loop
that reserves all memory at start-up and forbids cudaMalloc / cudaFree later
(both can synchronize the device), a runtime whose memory comes only from its
own pool, or an allocator hook that must not re-enter the allocator.  For
them the library keeps the FP32 scale scratch of the unfused sequence in a
fixed device array of its own.  These tests check that this entry point gives
the same bits as dq4_nested_unfused with caller-owned scratch, on calls in a
row (the shared array still holds the previous call's scales), and that it
refuses a problem larger than the array before anything runs.

This file is collected last on purpose: a stop-at-first-failure run has then
already run every other test.
"""

import numpy as np
import pytest
import torch

import dq4_inputs as gen

pytestmark = pytest.mark.gpu

DT = {"f16": (torch.float16, 0), "bf16": (torch.bfloat16, 1), "f32": (torch.float32, 2)}
LIMIT_BLOCKS = 4194304  # DQ4_STATIC_SCRATCH_BLOCKS in include/dq4.h


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_weight_dequantization_gb300 as dq
    return dq.get_lib()


def _dev(p):
    d = torch.device("cuda:0")
    return {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(d)
            for k in ("packed", "scale_codes", "nested_absmax", "scale_codebook",
                      "value_codebook")}


def _bits(t):
    return t.cpu().view(torch.int32 if t.dtype == torch.float32 else torch.int16).numpy()


def _call(lib, p, t, kind, scratch=None):
    dtype, code = DT[kind]
    out = torch.full((p.n,), float("nan"), dtype=dtype, device="cuda:0")
    stream = torch.cuda.current_stream().cuda_stream
    args = (t["packed"].data_ptr(), t["scale_codes"].data_ptr(), t["nested_absmax"].data_ptr(),
            t["scale_codebook"].data_ptr(), t["value_codebook"].data_ptr(), float(p.offset), p.n,
            p.blocksize, p.nested_blocksize, code, out.data_ptr())
    if scratch is None:
        st = lib.dq4_nested_unfused_static(*args, stream)
    else:
        st = lib.dq4_nested_unfused(*args, scratch.data_ptr(), stream)
    assert st == 0, lib.dq4_status_string(st)
    return out


def test_static_scratch_matches_caller_scratch_on_calls_in_a_row(lib):
    problems = [
        (gen.CELLS["C2a"].problem(), "bf16"),                                     # odd length
        (gen.make_problem(64 * 256 * 3 + 64 * 5 + 7, 32, 256, "fp4", 0.5, 0.52, seed=61), "f16"),
        (gen.make_problem(1 << 20, 4096, 1, "nf4", 1.0, -1e-3, seed=62), "f32"),
    ]
    problems.append(problems[0])  # the first again, after the array held other scales
    for p, kind in problems:
        t = _dev(p)
        scratch = torch.empty(-(-p.n // p.blocksize), dtype=torch.float32, device="cuda:0")
        want = _bits(_call(lib, p, t, kind, scratch))
        got = _bits(_call(lib, p, t, kind))
        assert np.array_equal(got, want), (p.n, p.blocksize, kind)


def test_largest_allowed_and_too_large(lib):
    # exactly at the limit: ceil(n / 32) == DQ4_STATIC_SCRATCH_BLOCKS
    p = gen.make_problem(32 * LIMIT_BLOCKS - 5, 32, 256, "nf4", 0.5, 0.0371, seed=63)
    t = _dev(p)
    scratch = torch.empty(LIMIT_BLOCKS, dtype=torch.float32, device="cuda:0")
    assert np.array_equal(_bits(_call(lib, p, t, "f16")), _bits(_call(lib, p, t, "f16", scratch)))
    # one block more is refused before anything is enqueued
    tiny = torch.zeros(16, dtype=torch.uint8, device="cuda:0")
    f = torch.zeros(256, dtype=torch.float32, device="cuda:0")
    st = lib.dq4_nested_unfused_static(tiny.data_ptr(), tiny.data_ptr(), f.data_ptr(),
                                       f.data_ptr(), f.data_ptr(), 0.0, 32 * LIMIT_BLOCKS + 1, 32,
                                       256, 0, f.data_ptr(), None)
    assert st == 10  # DQ4_ERR_TOO_LARGE
    torch.cuda.synchronize()
