"""Parity of the CUDA path with the CPU oracle: bit for bit, through the C ABI.

Every comparison is on raw output bits (FP16/BF16/FP32), since the method is
a deterministic elementwise map with a fixed rounding order ("Fuse nested
scale reconstruction into SM103 4-bit dequantization", bitsandbytes issue
#21, section "Correctness requirements": bitwise identity; no FMA).
"""

import ctypes

import numpy as np
import pytest
import torch

import dq4_inputs as gen
import oracle

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
ORACLE_THREADS = 16


@pytest.fixture(scope="module")
def dq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_weight_dequantization_gb300 as m
    return m


DEV = torch.device("cuda:0")


def to_dev(p):
    return {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(DEV)
            for k in ("packed", "scale_codes", "nested_absmax", "scale_codebook",
                      "value_codebook")}


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16).numpy().view(
        np.uint32 if t.dtype == torch.float32 else np.uint16)


def want_bits(arr: np.ndarray) -> np.ndarray:
    return arr.view(np.uint32) if arr.dtype == np.float32 else arr


def assert_same(got: torch.Tensor, want: np.ndarray, what: str):
    g = bits(got)
    w = want_bits(want)
    assert g.shape == w.shape, what
    if not np.array_equal(g, w):
        bad = np.flatnonzero(g != w)
        raise AssertionError(f"{what}: {bad.size} of {g.size} values differ; first at "
                             f"{bad[:5].tolist()}: got {[hex(int(x)) for x in g[bad[:5]]]} "
                             f"want {[hex(int(x)) for x in w[bad[:5]]]}")


def fused(dq, p, t, kind, **kw):
    """The fused entry point for problem p (device tensors t), output dtype name ``kind``."""
    return dq.dq4_nested(t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
                         t["value_codebook"], float(p.offset), p.n, p.blocksize,
                         p.nested_blocksize, DT[kind], **kw)


def unfused(dq, p, t, kind):
    return dq.dq4_nested_unfused(t["packed"], t["scale_codes"], t["nested_absmax"],
                                 t["scale_codebook"], t["value_codebook"], float(p.offset), p.n,
                                 p.blocksize, p.nested_blocksize, DT[kind])


# --------------------------------------------------------------- suites
def test_tail_suite_fused_unfused_plain(dq):
    """Odd lengths, packed tails, partial outer blocks and nested groups; all dtypes."""
    for name, p, out in gen.tail_suite():
        t = to_dev(p)
        want = oracle.dq4_nested(p, out, threads=ORACLE_THREADS)
        assert_same(fused(dq, p, t, out), want, name + " fused")
        res, scratch = unfused(dq, p, t, out)
        assert_same(res, want, name + " unfused")
        scales = oracle.nested_scales(p)
        assert np.array_equal(bits(scratch)[:p.nblocks], scales.view(np.uint32)), name
        plain = dq.dq4(t["packed"], torch.from_numpy(scales).to(DEV), t["value_codebook"], p.n,
                       p.blocksize, DT[out])
        assert_same(plain, want, name + " non-nested")


@pytest.mark.parametrize("name", ["C1", "C2a", "C2b", "C3a", "C3b", "C3c", "C3d"])
def test_cells(dq, name):
    cell = gen.CELLS[name]
    p = cell.problem()
    t = to_dev(p)
    want = oracle.dq4_nested(p, cell.out, threads=ORACLE_THREADS)
    assert_same(fused(dq, p, t, cell.out), want, name)
    assert_same(unfused(dq, p, t, cell.out)[0], want, name + " unfused")


@pytest.mark.parametrize("name", ["C4a", "C4b", "C4c", "C4d"])
def test_large_weight_cells_full(dq, name):
    """28672x8192 (234,881,024 values), every output compared; C4a is the benchmarked case."""
    cell = gen.CELLS[name]
    p = cell.problem()
    t = to_dev(p)
    got = fused(dq, p, t, cell.out)
    want = oracle.dq4_nested(p, cell.out, threads=ORACLE_THREADS)
    assert_same(got, want, name)


def test_blocksize_sweep_all_cells(dq):
    """8192x8192 FP4-style, FP32, blocksize 32..4096 x offsets {-1, -1e-3, +1e-3, +1}."""
    names = [k for k in gen.CELLS if k.startswith("C5-")]
    assert len(names) == 32
    for name in names:
        cell = gen.CELLS[name]
        p = cell.problem()
        t = to_dev(p)
        want = oracle.dq4_nested(p, cell.out, threads=ORACLE_THREADS)
        assert_same(fused(dq, p, t, cell.out), want, name)
        del t


@pytest.mark.parametrize("offset", [1.0, -1.0, 1e-3, -1e-3, 0.0371, -0.0371, 0.52, -0.52])
@pytest.mark.parametrize("bs", [32, 4096])
def test_every_scale_code_and_nibble(dq, offset, bs):
    p = gen.enumeration_problem(offset, blocksize=bs)
    t = to_dev(p)
    for out in DT:
        assert_same(fused(dq, p, t, out), oracle.dq4_nested(p, out), f"enum {offset} {out}")


def test_hand_worked_golden_cases(dq):
    from tests.test_oracle_pins import _hand_problem, _load_cases
    for case in _load_cases():
        p = _hand_problem(case)
        t = to_dev(p)
        for out in DT:
            if "expected_values" in case:
                want = np.array([int(h, 16) for h in case["expected_values"][out]])
            else:
                want = np.full(p.n, int(case["expected"][out], 16))
            got = bits(fused(dq, p, t, out)).astype(np.int64)
            assert np.array_equal(got, want), (case["name"], out)


def test_nested_blocksizes_other_than_256(dq):
    for nbs in (1, 2, 64, 1024):
        p = gen.make_problem(64 * 4096 + 37, 64, nbs, "nf4", 1.0, -0.1, seed=77 + nbs)
        t = to_dev(p)
        for out in DT:
            assert_same(fused(dq, p, t, out), oracle.dq4_nested(p, out), f"nbs {nbs} {out}")


def test_max_size_beyond_2_pow_32_values(dq):
    """n = 2^32 + 4099 values (64-bit indexing, odd tail); oracle on windows.

    Windows start on nested-group boundaries so that the oracle sees exactly
    the sub-problem: the first, one across value 2^31 and 2^32, and the last.
    """
    n = (1 << 32) + 4099
    p = gen.make_problem(n, 64, 256, "nf4", 0.5, 0.0371, seed=4242)
    t = to_dev(p)
    out = fused(dq, p, t, "f16")
    torch.cuda.synchronize()
    unit = 64 * 256
    for lo in (0, (1 << 31) - 2 * unit, (1 << 32) - 2 * unit, (n // unit) * unit - unit):
        hi = min(n, lo + 4 * unit)
        sub = gen.Problem(p.packed[lo // 2:(hi + 1) // 2], p.scale_codes[lo // 64:-(-hi // 64)],
                          p.nested_absmax[lo // unit:-(-hi // unit)], p.scale_codebook,
                          p.value_codebook, p.offset, hi - lo, 64, 256)
        assert_same(out[lo:hi], oracle.dq4_nested(sub, "f16"), f"window {lo}")
    del out, t
    torch.cuda.empty_cache()


# ------------------------------------------------- boundary properties
def test_output_canaries_untouched(dq):
    """Guard zones before and after the output are never written (odd tails included)."""
    guard = 4096
    for n in (1, 7, 8, 9, 4097 * 3, 64 * 256 + 1, 1 << 20):
        p = gen.make_problem(n, 64, 256, "fp4", 0.5, -0.52, seed=n)
        t = to_dev(p)
        for out in DT:
            isz = torch.empty(0, dtype=DT[out]).element_size()
            buf = torch.full(((n * isz + 2 * guard + 15) // 16 * 16,), 0xA5, dtype=torch.uint8,
                             device=DEV)
            view = buf[guard:guard + n * isz].view(DT[out])
            fused(dq, p, t, out, out=view)
            host = buf.cpu().numpy()
            assert np.all(host[:guard] == 0xA5) and np.all(host[guard + n * isz:] == 0xA5), (n, out)
            assert_same(view, oracle.dq4_nested(p, out), f"canary n={n} {out}")


def test_misaligned_pointers_take_the_per_value_path(dq):
    n = 64 * 777 + 13
    p = gen.make_problem(n, 64, 256, "nf4", 0.5, 0.1, seed=3)
    t = to_dev(p)
    packed_buf = torch.empty(p.packed.size + 1, dtype=torch.uint8, device=DEV)
    packed_buf[1:] = t["packed"]
    t2 = dict(t, packed=packed_buf[1:])
    for out in DT:
        out_buf = torch.empty(n + 1, dtype=DT[out], device=DEV)
        res = fused(dq, p, t2, out, out=out_buf[1:])
        assert_same(res, oracle.dq4_nested(p, out), f"misaligned {out}")


def test_repeated_launches_and_inputs_untouched(dq):
    p = gen.CELLS["C2a"].problem()
    t = to_dev(p)
    before = {k: v.clone() for k, v in t.items()}
    out = torch.empty(p.n, dtype=torch.bfloat16, device=DEV)
    for _ in range(3):
        fused(dq, p, t, "bf16", out=out)
    assert_same(out, oracle.dq4_nested(p, "bf16", threads=ORACLE_THREADS), "repeat")
    for k in t:
        assert torch.equal(before[k], t[k]), k


def test_stream_ordering(dq):
    """Work on a side stream: an H2D refill of the inputs, then the call, in stream order."""
    p1 = gen.make_problem(1 << 22, 64, 256, "nf4", 0.5, 0.0371, seed=1)
    p2 = gen.make_problem(1 << 22, 64, 256, "nf4", 0.5, 0.0371, seed=2)
    t = to_dev(p1)
    s = torch.cuda.Stream()
    host = torch.from_numpy(p2.packed.copy()).pin_memory()
    out = torch.empty(p1.n, dtype=torch.float16, device=DEV)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        torch.cuda._sleep(20_000_000)
        t["packed"].copy_(host, non_blocking=True)
        fused(dq, p1, t, "f16", out=out, stream=s)
    s.synchronize()
    p2.scale_codes, p2.nested_absmax = p1.scale_codes, p1.nested_absmax
    assert_same(out, oracle.dq4_nested(p2, "f16"), "stream order")


def test_cuda_graph_capture_and_replay(dq):
    p = gen.make_problem(1 << 20, 64, 256, "nf4", 0.5, 0.0371, seed=5)
    t = to_dev(p)
    out = torch.empty(p.n, dtype=torch.float16, device=DEV)
    fused(dq, p, t, "f16", out=out)  # first call fills the device cache outside capture
    torch.cuda.synchronize()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fused(dq, p, t, "f16", out=out, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert_same(out, oracle.dq4_nested(p, "f16"), "graph replay")


def test_n_zero_and_errors(dq):
    p = gen.make_problem(1000, 64, 256, "nf4", 0.5, 0.1, seed=9)
    t = to_dev(p)
    empty = torch.empty(0, dtype=torch.float16, device=DEV)
    z = dq.dq4_nested(t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
                      t["value_codebook"], 0.1, 0, 64, 256, torch.float16, out=empty)
    assert z.numel() == 0
    with pytest.raises(dq.Dq4Error, match="BLOCKSIZE"):
        dq.dq4_nested(t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
                      t["value_codebook"], 0.1, 1000, 8192, 256, torch.float16)
    L = dq.lib
    o = torch.empty(1000, dtype=torch.float16, device=DEV)
    st = L.dq4_nested(t["packed"].data_ptr(), t["scale_codes"].data_ptr(),
                      t["nested_absmax"].data_ptr(), t["scale_codebook"].data_ptr(),
                      t["value_codebook"].data_ptr(), 0.1, 1000, 64, 3, 0, o.data_ptr(), None)
    assert st == 4  # DQ4_ERR_NESTED_BLOCKSIZE
    st = L.dq4_nested(t["packed"].data_ptr(), t["scale_codes"].data_ptr(),
                      t["nested_absmax"].data_ptr() + 2, t["scale_codebook"].data_ptr(),
                      t["value_codebook"].data_ptr(), 0.1, 1000, 64, 256, 0,
                      torch.empty(1000, dtype=torch.float16, device=DEV).data_ptr(), None)
    assert st == 6  # DQ4_ERR_ALIGN


def test_gpu_conversions_through_the_kernel(dq):
    """RN16/RNbf16 of ~2M FP32 values (random and tie-adjacent), via the plain kernel.

    value_codebook[1] = 1.0 and every nibble is 1, so out = RN(1.0 * absmax[b])
    = RN(absmax[b]) exactly; compared with the oracle's converters.
    """
    rng = np.random.default_rng(17)
    u = rng.integers(0, 1 << 32, size=1 << 21, dtype=np.uint64).astype(np.uint32)
    u[: 1 << 19] = (u[: 1 << 19] & ~np.uint32(0x1FFF)) | np.uint32(0x1000)    # F16 ties
    u[1 << 19: 1 << 20] = (u[1 << 19: 1 << 20] & ~np.uint32(0xFFFF)) | np.uint32(0x8000)  # BF16
    x = u.view(np.float32)
    x = np.ascontiguousarray(x[np.isfinite(x)])
    bs = 32
    n = x.size * bs
    vcb = np.zeros(16, dtype=np.float32)
    vcb[1] = 1.0
    packed = torch.full((n // 2,), 0x11, dtype=torch.uint8, device=DEV)
    absmax = torch.from_numpy(x).to(DEV)
    vcb_d = torch.from_numpy(vcb).to(DEV)
    for out, conv in (("f16", oracle.f32_to_f16_bits), ("bf16", oracle.f32_to_bf16_bits)):
        got = bits(dq.dq4(packed, absmax, vcb_d, n, bs, DT[out])).reshape(-1, bs)
        assert np.all(got == got[:, :1])
        assert np.array_equal(got[:, 0], conv(x)), out


def test_gpu_conversions_exhaustive(dq):
    """Every FP32 bit pattern through the kernel's FP16 and BF16 conversions.

    value_codebook[1] = 1.0 and every nibble is 1, so each output is RN(absmax[b]): the
    2^32 patterns go in as absmax values, 2^25 per launch, and every one of a block's 32
    outputs must equal torch's conversion of that value on the same GPU (IEEE
    round-to-nearest-even, the rule the oracle's converters are pinned to over all 2^32
    inputs on the CPU).  NaN payloads are not specified, so NaN patterns are replaced by 0;
    infinities and values that overflow to infinity stay.
    """
    bs, chunk = 32, 1 << 25
    packed = torch.full((chunk * bs // 2,), 0x11, dtype=torch.uint8, device=DEV)
    vcb = torch.zeros(16, dtype=torch.float32, device=DEV)
    vcb[1] = 1.0
    bufs = {k: torch.empty(chunk * bs, dtype=DT[k], device=DEV) for k in ("f16", "bf16")}
    for start in range(0, 1 << 32, chunk):
        u = torch.arange(start, start + chunk, dtype=torch.int64, device=DEV).to(torch.int32)
        x = u.view(torch.float32)
        x = torch.where(torch.isnan(x), torch.zeros_like(x), x)
        for out, buf in bufs.items():
            dq.dq4(packed, x, vcb, chunk * bs, bs, DT[out], out=buf)
            want = x.to(DT[out]).view(torch.int16)
            got = buf.view(torch.int16).view(-1, bs)
            assert torch.equal(got, want.view(-1, 1).expand(-1, bs)), (out, hex(start))


def test_grid_stride_fallback_path(dq, tmp_path):
    """A build capped at one CTA per SM makes every warp loop over many tiles,
    loading the next tile before decoding the current one: same bits."""
    from quantized_weight_dequantization_gb300 import build as B
    path = B.build(force=True, out=str(tmp_path / "libdq4_capped.so"),
                   extra_flags=["-DDQ4_CTAS_PER_SM=1"])
    L = ctypes.CDLL(path)
    p_, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    L.dq4_nested.argtypes = [p_, p_, p_, p_, p_, f32, i64, i32, i32, i32, p_, p_]
    L.dq4_nested.restype = ctypes.c_int
    cases = [(gen.CELLS["C2a"].problem(), "bf16"), (gen.CELLS["C2b"].problem(), "f32")]
    cases += [(gen.enumeration_problem(-0.52, blocksize=32), k) for k in DT]
    cases += [(gen.make_problem(64 * 256 * 37 + 5, 4096, 256, "nf4", 0.5, 0.1, seed=8), k)
              for k in DT]
    for p, kind in cases:
        t = to_dev(p)
        out = torch.empty(p.n, dtype=DT[kind], device=DEV)
        st = L.dq4_nested(t["packed"].data_ptr(), t["scale_codes"].data_ptr(),
                          t["nested_absmax"].data_ptr(), t["scale_codebook"].data_ptr(),
                          t["value_codebook"].data_ptr(), float(p.offset), p.n, p.blocksize,
                          p.nested_blocksize, {"f16": 0, "bf16": 1, "f32": 2}[kind],
                          out.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == 0
        assert_same(out, oracle.dq4_nested(p, kind, threads=ORACLE_THREADS),
                    f"capped n={p.n} bs={p.blocksize} {kind}")
