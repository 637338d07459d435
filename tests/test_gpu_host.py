"""dq4_nested_host (host arrays in, host array out, pipelined by chunk) on the GPU.

Its values are dq4_nested's ("Fuse nested scale reconstruction into SM103
4-bit dequantization", bitsandbytes issue #21, section "Proposed
experiment"), so the checks are bit equality with the device path and with
the oracle, across chunk boundaries (small scratch buffers force many
chunks, the last one partial), dtypes, block sizes and pageable inputs.
"""

import numpy as np
import pytest
import torch

import dq4_inputs as gen
import oracle

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TDT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
KEYS = ("packed", "scale_codes", "nested_absmax", "scale_codebook", "value_codebook")


@pytest.fixture(scope="module")
def dq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_weight_dequantization_gb300 as m
    return m


def host_inputs(p, pin=True):
    t = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))) for k in KEYS}
    return {k: v.pin_memory() for k, v in t.items()} if pin else t


def device_result(dq, p, out):
    t = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(DEV) for k in KEYS}
    r = dq.dq4_nested(t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
                      t["value_codebook"], float(p.offset), p.n, p.blocksize,
                      p.nested_blocksize, TDT[out])
    return r.cpu()


def host_result(dq, p, out, scratch_groups=None, pin=True):
    h = host_inputs(p, pin)
    scratch = None
    if scratch_groups is not None:  # room for two buffers of `scratch_groups` nested groups
        group = p.blocksize * p.nested_blocksize
        need = int(dq.lib.dq4_nested_host_scratch_bytes(group * scratch_groups, p.blocksize,
                                                        p.nested_blocksize,
                                                        {"f16": 0, "bf16": 1, "f32": 2}[out]))
        scratch = torch.empty(need, dtype=torch.uint8, device=DEV)
    res = dq.dq4_nested_host(h["packed"], h["scale_codes"], h["nested_absmax"],
                             h["scale_codebook"], h["value_codebook"], float(p.offset), p.n,
                             p.blocksize, p.nested_blocksize, out_dtype=TDT[out], device=DEV,
                             scratch=scratch)
    torch.cuda.synchronize()
    return res


def bits(t):
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16).numpy()


@pytest.mark.parametrize("out", ["f16", "bf16", "f32"])
def test_many_chunks_equal_device_path(dq, out):
    # 37 whole nested groups and a partial one: 3-group chunks give 13 chunks
    n = 64 * 256 * 37 + 1234 + 1
    p = gen.make_problem(n, 64, 256, "nf4", 0.5, 0.0371, seed=5)
    got = host_result(dq, p, out, scratch_groups=3)
    assert np.array_equal(bits(got), bits(device_result(dq, p, out)))


@pytest.mark.parametrize("bs,nbs", [(32, 1), (4096, 2), (256, 64)])
def test_blocksizes_and_oracle(dq, bs, nbs):
    n = bs * nbs * 9 + 17
    p = gen.make_problem(n, bs, nbs, "fp4", 1.0, -0.5, seed=bs + nbs)
    got = host_result(dq, p, "f16", scratch_groups=2)
    assert np.array_equal(bits(got).view(np.uint16), oracle.dq4_nested(p, "f16"))


def test_default_scratch_pageable_inputs_and_tails(dq):
    """The tail suite's small problems (partial blocks, groups, odd lengths), pageable."""
    for name, p, out in gen.tail_suite():
        if p.n > 64 * 256 * 4:
            continue
        got = host_result(dq, p, out, pin=False)
        assert np.array_equal(bits(got), bits(device_result(dq, p, out))), name


def test_too_small_scratch_is_refused(dq):
    p = gen.make_problem(64 * 256 * 4, 64, 256, "nf4", 0.5, 0.0, seed=1)
    h = host_inputs(p)
    scratch = torch.empty(4096, dtype=torch.uint8, device=DEV)
    with pytest.raises(dq.Dq4Error, match="DQ4_ERR_TOO_LARGE"):
        dq.dq4_nested_host(h["packed"], h["scale_codes"], h["nested_absmax"],
                           h["scale_codebook"], h["value_codebook"], 0.0, p.n, 64, 256,
                           device=DEV, scratch=scratch)


def test_ordered_in_the_stream(dq):
    """The call's copies wait for work enqueued before it: here the copy that fills its
    host input from the device, held back behind a GPU sleep."""
    p = gen.make_problem(64 * 256 * 8, 64, 256, "nf4", 0.5, 0.0371, seed=9)
    h = host_inputs(p)
    real = h["packed"].to(DEV)
    h["packed"].zero_()  # stale until the stream's copy below runs
    s = torch.cuda.Stream(DEV)
    with torch.cuda.stream(s):
        torch.cuda._sleep(2_000_000)  # ~1 ms of GPU time ahead of the copy
        h["packed"].copy_(real, non_blocking=True)
        out = dq.dq4_nested_host(h["packed"], h["scale_codes"], h["nested_absmax"],
                                 h["scale_codebook"], h["value_codebook"], float(p.offset),
                                 p.n, 64, 256, device=DEV, stream=s)
    s.synchronize()
    assert np.array_equal(bits(out), bits(device_result(dq, p, "f16")))
