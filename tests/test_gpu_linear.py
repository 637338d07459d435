"""Nested 4-bit dequantization fused into a tcgen05 GEMM (Y = X W^T), on the GPU.

The dequantize-plus-linear path of "Fuse nested scale reconstruction into
SM103 4-bit dequantization" (bitsandbytes issue #21, sections "Problem" and
"B300 evidence plan") without the materialised weight.  Checks:
(1) integer-valued W (|w| <= 16) and ternary X: every FP32 partial sum is an
exact integer, so Y must equal the float64 oracle exactly (and its BF16/FP16
rounding exactly);
(2) realistic NF4 weights and normal activations within an FP32
accumulation bound, after the operand bits themselves are pinned by the
dequantization tests ("Correctness requirements": the dequantized tensor
passes bitwise equality before any GEMM tolerance).
"""

import numpy as np
import pytest
import torch

import dq4_inputs as gen
import oracle

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TDT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


@pytest.fixture(scope="module")
def dq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_weight_dequantization_gb300 as m
    return m


def run(dq, p, X, N, K, out=None, bad=None):
    t = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(DEV)
         for k in ("packed", "scale_codes", "nested_absmax", "scale_codebook", "value_codebook")}
    return dq.linear(X, t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
                     t["value_codebook"], float(p.offset), N, p.blocksize, p.nested_blocksize,
                     out_dtype=out, bad=bad)


def x_bits(X):
    return X.cpu().view(torch.int16).numpy().view(np.uint16)


def rounded(y64, out):
    t = torch.from_numpy(y64)
    return t.to(TDT[out]).to(torch.float64).numpy() if out != "f32" else \
        t.to(torch.float32).to(torch.float64).numpy()


# The kernel picks its activation-tile width BX from M, N, K and the SM count; on a
# 152-SM GB300 the shapes with N = 4860 take BX = 32, 64, 128 and 256 (38 weight tiles,
# the last one ragged), the others BX = 16 or 128; N = 4700 gives an odd count of
# weight tiles (37) at BX = 128 and 256.  Most run one CTA per tile; (128, 256, 4096)
# splits its units over the SMs.
SHAPES = [(1, 128, 64), (5, 200, 128), (127, 130, 192), (128, 256, 4096), (300, 1000, 512),
          (129, 384, 1024), (2048, 768, 256), (128, 4860, 192), (256, 4860, 128),
          (512, 4860, 64), (1024, 4860, 256), (512, 4700, 128), (2048, 4700, 64)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("xin", ["bf16", "f16"])
def test_integer_exact(dq, M, N, K, xin):
    p = gen.make_integer_problem(N, K, blocksize=64 if K % 64 == 0 else 32, seed=N + K)
    X = torch.from_numpy(gen.make_ternary_g(M, K, seed=M)).to(TDT[xin]).to(DEV)
    bad = torch.zeros(1, dtype=torch.int32, device=DEV)
    want = oracle.linear(p, x_bits(X), xin, N, K, threads=16)
    for out in ("f32", xin):
        got = run(dq, p, X, N, K, out=TDT[out], bad=bad).to(torch.float64).cpu().numpy()
        assert np.array_equal(got, rounded(want, out)), (M, N, K, xin, out,
                                                          np.abs(got - want).max())
    assert int(bad.item()) == 0


# With K a multiple of 256 the kernel reads each row's scale codes for four K
# steps in one aligned load of 256 / blocksize bytes (8, 4, 2 or 1) when one
# absmax group covers them; (32, 1) and (64, 2) take the per-K-step loads.
@pytest.mark.parametrize("bs,nbs", [(32, 1), (4096, 256), (64, 2), (32, 256), (128, 4),
                                    (256, 1), (64, 4)])
def test_blocksizes(dq, bs, nbs):
    M, N, K = 256, 512, 4096
    p = gen.make_integer_problem(N, K, blocksize=bs, nested_blocksize=nbs, seed=bs)
    X = torch.from_numpy(gen.make_ternary_g(M, K, seed=3)).to(torch.bfloat16).to(DEV)
    got = run(dq, p, X, N, K, out=torch.float32).double().cpu().numpy()
    assert np.array_equal(got, oracle.linear(p, x_bits(X), "bf16", N, K, threads=16))


def test_unaligned_scale_codes(dq):
    """Codes at an odd address: the per-K-step loads, same result."""
    M, N, K = 64, 384, 1024
    p = gen.make_integer_problem(N, K, seed=5)
    X = torch.from_numpy(gen.make_ternary_g(M, K, seed=6)).to(torch.bfloat16).to(DEV)
    t = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(DEV)
         for k in ("packed", "nested_absmax", "scale_codebook", "value_codebook")}
    buf = torch.zeros(p.scale_codes.size + 1, dtype=torch.uint8, device=DEV)
    codes = buf[1:]
    codes.copy_(torch.from_numpy(p.scale_codes))
    got = dq.linear(X, t["packed"], codes, t["nested_absmax"], t["scale_codebook"],
                    t["value_codebook"], 0.0, N, 64, 256, out_dtype=torch.float32)
    want = oracle.linear(p, x_bits(X), "bf16", N, K, threads=16)
    assert np.array_equal(got.double().cpu().numpy(), want)


@pytest.mark.parametrize("M", [16, 128, 512, 2048])
def test_realistic_llm_shape(dq, M):
    """An 11008 x 4096 NF4-style nested weight (blocksize 64, nested 256)."""
    N, K = 11008, 4096
    p = gen.make_problem(N * K, 64, 256, "nf4", 1.0, 0.0371, seed=21)
    X = torch.from_numpy(gen.make_normal_g(M, K, seed=22)).to(torch.bfloat16).to(DEV)
    bad = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = run(dq, p, X, N, K, out=torch.float32, bad=bad).double().cpu().numpy()
    xb = x_bits(X)
    want = oracle.linear(p, xb, "bf16", N, K, threads=16)
    w = oracle._bits16_to_f64(oracle.dq4_nested(p, "bf16", threads=16), "bf16").reshape(N, K)
    x = oracle._bits16_to_f64(xb, "bf16")
    norm = np.sqrt((x * x) @ (w * w).T)  # sqrt(sum_k (x_k w_k)^2) per entry
    tol = 16 * 2.0 ** -24 * K * norm + 1e-30
    err = np.abs(got - want)
    assert np.all(err <= tol), float((err / tol).max())
    assert int(bad.item()) == 0


def test_repeated_and_back_to_back(dq):
    M, N, K = 200, 700, 512
    p = gen.make_integer_problem(N, K, seed=9)
    X = torch.from_numpy(gen.make_ternary_g(M, K, seed=10)).to(torch.bfloat16).to(DEV)
    outs = [run(dq, p, X, N, K, out=torch.float32) for _ in range(4)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_errors(dq):
    p = gen.make_integer_problem(64, 100, blocksize=32, seed=1)
    X = torch.zeros((4, 100), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(dq.Dq4Error, match="DQ4_ERR_N"):
        run(dq, p, X, 64, 100)
    # packed is read by TMA: a base that is not 16-byte aligned is refused on the host
    p = gen.make_integer_problem(64, 128, seed=2)
    X = torch.zeros((4, 128), dtype=torch.bfloat16, device=DEV)
    t = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(DEV)
         for k in ("scale_codes", "nested_absmax", "scale_codebook", "value_codebook")}
    buf = torch.zeros(p.packed.size + 16, dtype=torch.uint8, device=DEV)
    packed = buf[4:4 + p.packed.size]
    with pytest.raises(dq.Dq4Error, match="DQ4_ERR_ALIGN"):
        dq.linear(X, packed, t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
                  t["value_codebook"], 0.0, 64, 64, 256)


# Tiles that would not fill the SMs in whole rounds: with a workspace one CTA per SM
# takes an equal share of the (tile, stage) units, a run that may cross tile boundaries;
# partial FP32 tiles are summed in K order by the last CTA to finish each tile.  On a
# 152-SM GB300 these take (BX, most tiles one CTA touches): (16, 2), (16, 1), (128, 2),
# (16, 1) with a partial last stage (K = 1216), (32, 2), (128, 2) ragged, (128, 3)
# ragged, (256, 2) ragged, (256, 3) with a partial last stage, (256, 4) ragged with
# one-stage tiles of one K step, (256, 5) one-stage, (16, 3), (256, 5), and (64, 2)
# twice (M = 64 and a ragged M = 40).  BX <= 64 issues its MMAs from two threads, each
# into its own accumulators (two buffers each up to BX = 32, one at BX = 64); wider tiles
# issue from one thread into one buffer.
SPLIT_SHAPES = [(16, 11008, 4096), (3, 2000, 4096), (640, 1024, 8192), (16, 4860, 1216),
                (128, 2000, 2048), (200, 3000, 8192), (300, 9856, 2048), (300, 9856, 4096),
                (1024, 9856, 1216), (1500, 9856, 64), (2048, 9856, 256), (16, 49152, 512),
                (2048, 9856, 512), (64, 2000, 16384), (40, 2000, 16384)]


@pytest.mark.parametrize("M,N,K", SPLIT_SHAPES)
def test_split_and_whole_tiles_are_exact(dq, M, N, K):
    assert dq.lib.dq4_nested_linear_workspace_bytes(M, N, K) > 0  # the split path applies
    p = gen.make_integer_problem(N, K, seed=M + N)
    X = torch.from_numpy(gen.make_ternary_g(M, K, seed=K)).to(torch.bfloat16).to(DEV)
    want = oracle.linear(p, x_bits(X), "bf16", N, K, threads=16)
    t = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(DEV)
         for k in ("packed", "scale_codes", "nested_absmax", "scale_codebook", "value_codebook")}
    none = torch.empty(0, dtype=torch.uint8, device=DEV)
    for ws in (None, none):  # cached workspace (split) / no workspace (whole tiles)
        bad = torch.zeros(1, dtype=torch.int32, device=DEV)
        got = dq.linear(X, t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
                        t["value_codebook"], 0.0, N, 64, 256, out_dtype=torch.float32, bad=bad,
                        workspace=ws)
        assert np.array_equal(got.double().cpu().numpy(), want), (M, N, K, ws is None)
        assert int(bad.item()) == 0


def test_split_workspace_is_left_zero_and_reusable(dq):
    M, N, K = 16, 4096, 2048
    need = int(dq.lib.dq4_nested_linear_workspace_bytes(M, N, K))
    assert need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    p = gen.make_integer_problem(N, K, seed=77)
    X = torch.from_numpy(gen.make_ternary_g(M, K, seed=78)).to(torch.bfloat16).to(DEV)
    t = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(DEV)
         for k in ("packed", "scale_codes", "nested_absmax", "scale_codebook", "value_codebook")}
    want = oracle.linear(p, x_bits(X), "bf16", N, K, threads=16)
    for _ in range(20):  # back to back on one stream, one workspace
        got = dq.linear(X, t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
                        t["value_codebook"], 0.0, N, 64, 256, out_dtype=torch.float32,
                        workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(got.double().cpu().numpy(), want)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    counts = ws[:4 * sms].view(torch.int32)  # the counters: one per SM, first
    assert int(counts.abs().sum().item()) == 0


def test_split_realistic_matches_whole_tiles(dq):
    """NF4 weights, normal activations: both paths within the FP32 bound, and the split
    path is deterministic (its partial sums meet in a fixed order)."""
    M, N, K = 16, 11008, 4096
    p = gen.make_problem(N * K, 64, 256, "nf4", 1.0, 0.0371, seed=23)
    X = torch.from_numpy(gen.make_normal_g(M, K, seed=24)).to(torch.bfloat16).to(DEV)
    t = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(DEV)
         for k in ("packed", "scale_codes", "nested_absmax", "scale_codebook", "value_codebook")}
    args = (X, t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
            t["value_codebook"], float(p.offset), N, 64, 256)
    split = [dq.linear(*args, out_dtype=torch.float32) for _ in range(3)]
    whole = dq.linear(*args, out_dtype=torch.float32,
                      workspace=torch.empty(0, dtype=torch.uint8, device=DEV))
    torch.cuda.synchronize()
    assert torch.equal(split[0], split[1]) and torch.equal(split[0], split[2])
    xb = x_bits(X)
    want = oracle.linear(p, xb, "bf16", N, K, threads=16)
    w = oracle._bits16_to_f64(oracle.dq4_nested(p, "bf16", threads=16), "bf16").reshape(N, K)
    x = oracle._bits16_to_f64(xb, "bf16")
    tol = 16 * 2.0 ** -24 * K * np.sqrt((x * x) @ (w * w).T) + 1e-30
    for got in (split[0], whole):
        assert np.all(np.abs(got.double().cpu().numpy() - want) <= tol)


def test_one_workspace_across_shapes(dq):
    """A workspace first used by a problem with few tiles, then by ones with more."""
    shapes = [(128, 256, 4096), (16, 11008, 1024), (300, 4096, 4096), (100, 2000, 512),
              (3, 2000, 4096), (2048, 9856, 512)]
    need = max(int(dq.lib.dq4_nested_linear_workspace_bytes(*sh)) for sh in shapes)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    for M, N, K in shapes + shapes[::-1]:
        p = gen.make_integer_problem(N, K, seed=M * 7 + K)
        X = torch.from_numpy(gen.make_ternary_g(M, K, seed=N)).to(torch.bfloat16).to(DEV)
        t = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(DEV)
             for k in ("packed", "scale_codes", "nested_absmax", "scale_codebook",
                       "value_codebook")}
        got = dq.linear(X, t["packed"], t["scale_codes"], t["nested_absmax"],
                        t["scale_codebook"], t["value_codebook"], 0.0, N, 64, 256,
                        out_dtype=torch.float32, workspace=ws)
        want = oracle.linear(p, x_bits(X), "bf16", N, K, threads=16)
        assert np.array_equal(got.double().cpu().numpy(), want), (M, N, K)


def test_workspace_is_bounded_by_the_sm_count(dq):
    """Partial tiles are kept per CTA (two each, one CTA per SM), not per tile."""
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    bound = (4 * sms + 255) // 256 * 256 + sms * 2 * 256 * 128 * 4
    for M, N, K in [(16, 11008, 4096), (512, 11008, 4096), (4096, 11008, 4096),
                    (4096, 28672, 8192), (65536, 4096, 4096)]:
        assert 0 <= int(dq.lib.dq4_nested_linear_workspace_bytes(M, N, K)) <= bound


@pytest.mark.parametrize("xin,out", [("f16", "f16"), ("f16", "f32"), ("bf16", "bf16")])
def test_split_dtypes_exact(dq, xin, out):
    """The split path with FP16 activations (the weight decoded to FP16) and 16-bit outputs."""
    M, N, K = 16, 4860, 2048
    assert dq.lib.dq4_nested_linear_workspace_bytes(M, N, K) > 0
    p = gen.make_integer_problem(N, K, seed=31)
    X = torch.from_numpy(gen.make_ternary_g(M, K, seed=32)).to(TDT[xin]).to(DEV)
    want = oracle.linear(p, x_bits(X), xin, N, K, threads=16)
    got = run(dq, p, X, N, K, out=TDT[out]).to(torch.float64).cpu().numpy()
    assert np.array_equal(got, rounded(want, out))


def test_graph_capture_and_replay(dq):
    """dq.linear captured in a CUDA graph (split path, cached workspace) replays exactly."""
    M, N, K = 16, 4096, 2048
    assert dq.lib.dq4_nested_linear_workspace_bytes(M, N, K) > 0
    p = gen.make_integer_problem(N, K, seed=41)
    t = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(DEV)
         for k in ("packed", "scale_codes", "nested_absmax", "scale_codebook", "value_codebook")}
    X = torch.zeros((M, K), dtype=torch.bfloat16, device=DEV)
    Y = torch.empty((M, N), dtype=torch.float32, device=DEV)
    call = lambda: dq.linear(X, t["packed"], t["scale_codes"], t["nested_absmax"],
                             t["scale_codebook"], t["value_codebook"], 0.0, N, 64, 256, Y=Y)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call()  # the workspace for (device, stream) exists before capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            call()
    for seed in (1, 2, 3):
        G = gen.make_ternary_g(M, K, seed=seed)
        X.copy_(torch.from_numpy(G).to(torch.bfloat16))
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        want = oracle.linear(p, x_bits(X), "bf16", N, K, threads=16)
        assert np.array_equal(Y.double().cpu().numpy(), want), seed


# ---- the decoded weight operand itself, bit for bit ("Correctness requirements": the
# dequantized tensor passes bitwise equality before any GEMM tolerance).  Activation rows
# that are unit vectors e_k make each entry of Y = X W^T one weight, w[n, k] * 1, plus
# products with exact zeros: the FP32 accumulator holds w exactly whatever the summation
# order, so Y^T must equal dq4_nested's output for X's dtype bit for bit.  The one thing a
# GEMM cannot show is the sign of a zero weight (its +0 and -0 terms may sum to +0), so a
# zero weight must give a zero of either sign.  Every k is covered at every M below, so
# every activation-tile width the planner picks decodes the whole weight, on the split
# path (cached workspace) and on whole tiles (no workspace).
OPERAND_CASES = [
    # fmt, absmax sigma, offset, blocksize, nested blocksize, X dtype, N, K, Ms
    ("nf4", 1.0, 0.0371, 64, 256, "bf16", 11008, 4096, (16, 32, 64, 128, 256, 4096)),
    ("fp4", 0.5, -0.52, 64, 256, "f16", 11008, 4096, (16, 32, 64, 128, 256, 4096)),
    ("nf4", 0.5, -0.0371, 32, 256, "f16", 4860, 1216, (16, 64, 1216)),    # per-K-step codes
    ("fp4", 1.0, 0.52, 4096, 256, "bf16", 4700, 2048, (16, 128, 2048)),  # blocks span rows
    ("nf4", 0.5, 0.52, 128, 256, "bf16", 2000, 4096, (32, 256)),
    ("fp4", 0.5, -0.0371, 1024, 1, "f16", 3000, 1024, (16, 64, 1024)),
    ("nf4", 1.0, -0.52, 256, 64, "bf16", 1111, 2048, (48, 300)),
]


def _f32_bits_of(bits16: np.ndarray, xin: str) -> np.ndarray:
    """FP32 bit patterns of 16-bit values (both conversions are exact)."""
    if xin == "bf16":
        return (bits16.astype(np.uint32) << 16).view(np.int32)
    return bits16.view(np.float16).astype(np.float32).view(np.int32)


def _nonzero_bits(t: torch.Tensor, int_dtype) -> torch.Tensor:
    """Raw bits with both zeros mapped to +0 (float view t, integer view of the same width)."""
    return torch.where(t == 0, torch.zeros((), dtype=int_dtype, device=t.device),
                       t.view(int_dtype))


@pytest.mark.parametrize("case", OPERAND_CASES, ids=lambda c: f"{c[0]}-bs{c[3]}-nbs{c[4]}-"
                         f"{c[5]}-{c[6]}x{c[7]}")
def test_weight_operand_bits_with_unit_activations(dq, case):
    fmt, sigma, offset, bs, nbs, xin, N, K, Ms = case
    p = gen.make_problem(N * K, bs, nbs, fmt, sigma, offset, seed=N + bs + nbs)
    w16 = oracle.dq4_nested(p, xin, threads=16)
    want32 = torch.from_numpy(_f32_bits_of(w16, xin).reshape(N, K)).to(DEV).t().contiguous()
    want16 = torch.from_numpy(w16.view(np.int16).reshape(N, K)).to(DEV).t().contiguous()
    want32 = torch.where(want32.view(torch.float32) == 0, torch.zeros_like(want32), want32)
    want16 = _nonzero_bits(want16.view(TDT[xin]), torch.int16)
    t = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(DEV)
         for k in ("packed", "scale_codes", "nested_absmax", "scale_codebook", "value_codebook")}
    order = torch.from_numpy(np.argsort(gen.splitmix64(K, 77, K), kind="stable")).to(DEV)
    none = torch.empty(0, dtype=torch.uint8, device=DEV)
    split_seen = False
    for M in Ms:
        split_seen |= dq.lib.dq4_nested_linear_workspace_bytes(M, N, K) > 0
        for ws in (None, none):  # cached workspace (split when it pays) / whole tiles
            bad = torch.zeros(1, dtype=torch.int32, device=DEV)
            Yt = torch.empty((K, N), dtype=torch.float32, device=DEV)
            Yt16 = torch.empty((K, N), dtype=TDT[xin], device=DEV)
            for k0 in range(0, K, M):
                ks = order[k0:k0 + M]  # M distinct k (the last slice may be shorter)
                X = torch.zeros((ks.numel(), K), dtype=TDT[xin], device=DEV)
                X[torch.arange(ks.numel(), device=DEV), ks] = 1
                args = (X, t["packed"], t["scale_codes"], t["nested_absmax"],
                        t["scale_codebook"], t["value_codebook"], float(p.offset), N, bs, nbs)
                Yt[ks] = dq.linear(*args, out_dtype=torch.float32, bad=bad, workspace=ws)
                Yt16[ks] = dq.linear(*args, out_dtype=TDT[xin], bad=bad, workspace=ws)
            torch.cuda.synchronize()
            got32 = _nonzero_bits(Yt, torch.int32)
            got16 = _nonzero_bits(Yt16, torch.int16)
            ne = int((got32 != want32).sum().item())
            assert ne == 0, (M, ws is None, ne)
            assert torch.equal(got16, want16), (M, ws is None)
            assert int(bad.item()) == 0
    if N == 11008:
        assert split_seen  # the decode sizes take the split path at this shape


def test_weight_operand_bits_beyond_2_pow_31_values(dq):
    """N x K > 2^31 weight values (64-bit weight indices; a partial last row tile): 16 unit
    activation rows pick 16 columns k of W (the first, the last and 14 others), and those
    columns of every row in three windows (the first rows, the rows across flat index 2^31,
    the last rows) must equal dq4_nested's bits for X's dtype, on the split path (cached
    workspace) and on whole tiles (no workspace).  Zeros compare as zeros of either sign."""
    N, K, bs, nbs, xin = 65600, 32768, 64, 256, "bf16"
    assert N * K > (1 << 31)
    p = gen.make_problem(N * K, bs, nbs, "nf4", 1.0, 0.0371, seed=N + K)
    t = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(DEV)
         for k in ("packed", "scale_codes", "nested_absmax", "scale_codebook", "value_codebook")}
    perm = np.argsort(gen.splitmix64(K, 91, K), kind="stable")
    ks = [0, K - 1] + [int(k) for k in perm if k not in (0, K - 1)][:14]
    X = torch.zeros((len(ks), K), dtype=TDT[xin], device=DEV)
    X[torch.arange(len(ks), device=DEV), torch.tensor(ks, device=DEV)] = 1
    none = torch.empty(0, dtype=torch.uint8, device=DEV)
    args = (X, t["packed"], t["scale_codes"], t["nested_absmax"], t["scale_codebook"],
            t["value_codebook"], float(p.offset), N, bs, nbs)
    unit = bs * nbs
    mid = (1 << 31) // K  # the first row at flat index >= 2^31
    windows = [(0, 256), (mid - 64, mid + 32), (N - 96, N)]
    for ws in (None, none):
        bad = torch.zeros(1, dtype=torch.int32, device=DEV)
        Y = dq.linear(*args, out_dtype=torch.float32, bad=bad, workspace=ws)
        torch.cuda.synchronize()
        assert int(bad.item()) == 0
        for n0, n1 in windows:
            lo, hi = n0 * K, n1 * K  # K is a multiple of bs * nbs: whole nested groups
            assert lo % unit == 0 and hi % unit == 0
            sub = gen.Problem(p.packed[lo // 2:hi // 2], p.scale_codes[lo // bs:hi // bs],
                              p.nested_absmax[lo // unit:hi // unit], p.scale_codebook,
                              p.value_codebook, p.offset, hi - lo, bs, nbs)
            w16 = oracle.dq4_nested(sub, xin, threads=16).reshape(n1 - n0, K)[:, ks]
            want = torch.from_numpy(np.ascontiguousarray(_f32_bits_of(w16, xin).T)).to(DEV)
            want = torch.where(want.view(torch.float32) == 0, torch.zeros_like(want), want)
            got = _nonzero_bits(Y[:, n0:n1].contiguous(), torch.int32)
            ne = int((got != want).sum().item())
            assert ne == 0, (ws is None, n0, ne)
        del Y
    del t
    torch.cuda.empty_cache()
