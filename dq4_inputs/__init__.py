"""Seeded synthetic inputs for nested 4-bit dequantization.

This module builds the *inputs* of the method (packed nibbles, uint8 scale
codes, FP32 nested absmax, the two codebooks, the offset) and nothing else.
It holds none of the method's arithmetic: it never rebuilds a scale, decodes
a nibble or rounds to an output dtype.  Both the CPU oracle and the CUDA path
are fed from here, so that the two see the same bytes.

Randomness comes from splitmix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014): the k-th word of stream
``(seed, stream)`` is ``mix(base + k * 0x9E3779B97F4A7C15)``, with ``base``
itself a mixed function of ``seed`` and ``stream``.  Everything is
vectorised in numpy uint64 arithmetic, which wraps modulo 2**64.
"""

from __future__ import annotations

import dataclasses
import statistics
from typing import Optional

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# stream ids: every buffer draws from its own splitmix64 stream
STREAM_PACKED = 1
STREAM_CODES = 2
STREAM_ABSMAX = 3
STREAM_PLAIN_ABSMAX = 4


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, stream: int, count: int, start: int = 0) -> np.ndarray:
    """Words ``start .. start+count-1`` of the splitmix64 sequence for (seed, stream)."""
    with np.errstate(over="ignore"):
        base = _mix(np.array([(seed * 0x100000001B3 + stream) & 0xFFFFFFFFFFFFFFFF],
                             dtype=np.uint64))[0]
        k = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix(base + k * GOLDEN)


def uniform_bytes(seed: int, stream: int, nbytes: int, chunk_words: int = 1 << 24) -> np.ndarray:
    """``nbytes`` uniform random bytes (the little-endian bytes of the words).

    Generated in chunks of ``chunk_words`` words so that huge buffers need
    little memory beyond the result itself; the bytes do not depend on it.
    """
    nwords = (nbytes + 7) // 8
    res = np.empty(nwords * 8, dtype=np.uint8)
    words = res.view(np.uint64)
    for lo in range(0, nwords, chunk_words):
        hi = min(nwords, lo + chunk_words)
        words[lo:hi] = splitmix64(seed, stream, hi - lo, start=lo)
    return res[:nbytes]


def uniform_open01(words: np.ndarray) -> np.ndarray:
    """Map uint64 words to float64 uniforms in (0, 1] using the top 53 bits."""
    return ((words >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def lognormal_f32(seed: int, stream: int, count: int, sigma: float) -> np.ndarray:
    """``count`` FP32 samples of exp(sigma * z), z standard normal (Box-Muller, float64)."""
    w = splitmix64(seed, stream, 2 * count)
    u1 = uniform_open01(w[0::2])
    u2 = uniform_open01(w[1::2])
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return np.exp(sigma * z).astype(np.float32)


# ---------------------------------------------------------------- codebooks
def scale_codebook() -> np.ndarray:
    """256 sorted FP32 entries in [-1, 1]: ((2k - 255) / 255)^3 rounded once to FP32.

    Odd-symmetric, endpoints exactly +-1, strictly increasing, with magnitudes
    down to ~6e-8 so that cancellation against the offset is exercised.
    """
    x = (2.0 * np.arange(256, dtype=np.float64) - 255.0) / 255.0
    return (x * x * x).astype(np.float32)


def nf4_style_codebook() -> np.ndarray:
    """16 sorted FP32 entries with 0 and +-1: normal quantiles, 8 positive, 7 negative.

    Our own construction in the spirit of a normal-float table (it is not any
    library's table): positive j/8 and negative j/7 quantile steps of a
    standard normal over (0.5, 0.95], scaled so that the outermost are +-1.
    """
    nd = statistics.NormalDist()
    top = nd.inv_cdf(0.95)
    pos = [nd.inv_cdf(0.5 + 0.45 * j / 8) / top for j in range(1, 9)]
    neg = [-nd.inv_cdf(0.5 + 0.45 * j / 7) / top for j in range(1, 8)]
    vals = sorted(neg + [0.0] + pos)
    vals[0], vals[-1] = -1.0, 1.0  # exact endpoints
    return np.array(vals, dtype=np.float32)


def fp4_style_codebook() -> np.ndarray:
    """16 sorted FP32 entries: E2M1 magnitudes {0,.5,1,1.5,2,3,4,6}/6, both signs, -0 before +0."""
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64) / 6.0
    neg = (-mags[::-1]).astype(np.float32)  # ends with -0.0
    pos = mags.astype(np.float32)           # starts with +0.0
    cb = np.concatenate([neg, pos])
    assert np.signbit(cb[7]) and not np.signbit(cb[8])
    return cb


VALUE_CODEBOOKS = {"nf4": nf4_style_codebook, "fp4": fp4_style_codebook}

OUT_DTYPES = {"f16": 0, "bf16": 1, "f32": 2}
OUT_ITEMSIZE = {"f16": 2, "bf16": 2, "f32": 4}


# --------------------------------------------------------------- problems
@dataclasses.dataclass
class Problem:
    """All inputs of one nested dequantization call (host numpy arrays)."""

    packed: np.ndarray          # uint8[ceil(n/2)], high nibble = even index
    scale_codes: np.ndarray     # uint8[NB]
    nested_absmax: np.ndarray   # float32[NG]
    scale_codebook: np.ndarray  # float32[256]
    value_codebook: np.ndarray  # float32[16]
    offset: np.float32
    n: int
    blocksize: int
    nested_blocksize: int

    @property
    def nblocks(self) -> int:
        return -(-self.n // self.blocksize)

    @property
    def ngroups(self) -> int:
        return -(-self.nblocks // self.nested_blocksize)


def sizes(n: int, blocksize: int, nested_blocksize: int):
    """(packed bytes, NB, NG) for a problem of n values."""
    nb = -(-n // blocksize)
    return (n + 1) // 2, nb, -(-nb // nested_blocksize)


def make_problem(n: int, blocksize: int = 64, nested_blocksize: int = 256, fmt: str = "nf4",
                 sigma: float = 0.5, offset: float = 0.0371, seed: int = 0,
                 force_all_codes: bool = False) -> Problem:
    """Uniform random codes and lognormal(0, sigma) nested absmax from ``seed``.

    ``force_all_codes`` overwrites the first 256 scale codes with 0..255 and the
    first 16 values of every block with nibbles 0..15 (every code present).
    The padding nibble of an odd-length tail is left random on purpose.
    """
    npk, nb, ng = sizes(n, blocksize, nested_blocksize)
    packed = uniform_bytes(seed, STREAM_PACKED, npk)
    codes = uniform_bytes(seed, STREAM_CODES, nb)
    absmax = lognormal_f32(seed, STREAM_ABSMAX, ng, sigma)
    if force_all_codes:
        k = min(256, nb)
        codes[:k] = np.arange(k, dtype=np.uint8)
        # nibbles 0..15 at values b*bs + 0..15: bytes b*bs/2 + 0..7 = (2j)<<4 | (2j+1)
        pattern = np.array([(2 * j) << 4 | (2 * j + 1) for j in range(8)], dtype=np.uint8)
        starts = np.arange(nb, dtype=np.int64) * (blocksize // 2)
        for j in range(8):
            idx = starts + j
            idx = idx[2 * idx + 1 < n]  # both nibbles of the byte are real values
            packed[idx] = pattern[j]
    return Problem(packed=packed, scale_codes=codes, nested_absmax=absmax,
                   scale_codebook=scale_codebook(), value_codebook=VALUE_CODEBOOKS[fmt](),
                   offset=np.float32(offset), n=n, blocksize=blocksize,
                   nested_blocksize=nested_blocksize)


def make_plain_absmax(n: int, blocksize: int, seed: int, sigma: float = 0.5) -> np.ndarray:
    """FP32 per-block absmax for the non-nested form, lognormal(0, sigma)."""
    nb = -(-n // blocksize)
    return lognormal_f32(seed, STREAM_PLAIN_ABSMAX, nb, sigma)


# ------------------------------------------------------------------ cells
@dataclasses.dataclass(frozen=True)
class Cell:
    """One named workload: shape, format, block sizes, distribution, offset, output."""

    name: str
    rows: int
    cols: int
    fmt: str
    blocksize: int
    nested_blocksize: int
    sigma: float
    offset: float
    out: str
    seed: int
    force_all_codes: bool = False

    @property
    def n(self) -> int:
        return self.rows * self.cols

    def problem(self) -> Problem:
        return make_problem(self.n, self.blocksize, self.nested_blocksize, self.fmt,
                            self.sigma, self.offset, self.seed, self.force_all_codes)

    def algorithmic_bytes(self) -> int:
        """Bytes the method must move: inputs read once plus the output written once."""
        npk, nb, ng = sizes(self.n, self.blocksize, self.nested_blocksize)
        return npk + nb + 4 * ng + 4 * 256 + 4 * 16 + OUT_ITEMSIZE[self.out] * self.n


def _cells():
    cells = [
        # 4096x4096 NF4-style, FP16 out
        Cell("C1", 4096, 4096, "nf4", 64, 256, 0.5, 0.0371, "f16", 101),
        # odd-length tail control, FP4-style, BF16 and FP32 out
        Cell("C2a", 4097, 4095, "fp4", 64, 256, 0.5, -0.52, "bf16", 201),
        Cell("C2b", 4097, 4095, "fp4", 64, 256, 0.5, -0.52, "f32", 201),
        # LLM-shaped 11008x4096 / 4096x11008, NF4-style, BF16, lognormal(0, 1), offset +-0.1
        Cell("C3a", 11008, 4096, "nf4", 64, 256, 1.0, 0.1, "bf16", 301),
        Cell("C3b", 11008, 4096, "nf4", 64, 256, 1.0, -0.1, "bf16", 302),
        Cell("C3c", 4096, 11008, "nf4", 64, 256, 1.0, 0.1, "bf16", 303),
        Cell("C3d", 4096, 11008, "nf4", 64, 256, 1.0, -0.1, "bf16", 304),
        # large weight 28672x8192, NF4/FP4-style, FP16/BF16
        Cell("C4a", 28672, 8192, "nf4", 64, 256, 0.5, 0.0371, "f16", 401),
        Cell("C4b", 28672, 8192, "nf4", 64, 256, 0.5, 0.0371, "bf16", 402),
        Cell("C4c", 28672, 8192, "fp4", 64, 256, 0.5, 0.0371, "f16", 403),
        Cell("C4d", 28672, 8192, "fp4", 64, 256, 0.5, 0.0371, "bf16", 404),
    ]
    # blocksize sweep on 8192x8192, FP4-style, FP32 out, every code present
    seed = 501
    for bs in (32, 64, 128, 256, 512, 1024, 2048, 4096):
        for off in (-1.0, -1e-3, 1e-3, 1.0):
            cells.append(Cell(f"C5-bs{bs}-off{off:+g}", 8192, 8192, "fp4", bs, 256, 0.5, off,
                              "f32", seed, force_all_codes=True))
            seed += 1
    return {c.name: c for c in cells}


CELLS = _cells()


def tail_suite():
    """Small problems with partial outer blocks, partial nested groups and odd tails.

    Yields (name, Problem, out) triples.
    """
    ns = [1, 2, 3, 31, 33, 63, 65, 64 * 256 + 1, 64 * 256 * 3 + 64 * 5 + 7, 4097 * 4095]
    seed = 900
    for n in ns:
        for bs in (32, 64, 4096):
            for fmt, off in (("nf4", 0.52), ("fp4", -0.52)):
                for out in ("f16", "bf16", "f32"):
                    if n > 1 << 20 and (bs != 64 or out == "f32"):
                        continue  # keep the big odd case to one blocksize and two dtypes
                    p = make_problem(n, bs, 256, fmt, 0.5, off, seed)
                    yield f"T-n{n}-bs{bs}-{fmt}-{out}", p, out
                    seed += 1


def enumeration_problem(offset: float, blocksize: int = 32, groups: int = 4,
                        seed: int = 7) -> Problem:
    """Every (scale code, nibble) pair, in every one of ``groups`` nested groups.

    Block b uses scale code b mod 256 and its values run through nibbles
    0..15 repeatedly, so each group of 256 blocks covers the 256 x 16 grid.
    """
    nbs = 256
    nb = nbs * groups
    n = nb * blocksize
    codes = (np.arange(nb) % 256).astype(np.uint8)
    nib = np.arange(n) % 16
    packed = ((nib[0::2] << 4) | nib[1::2]).astype(np.uint8)
    absmax = lognormal_f32(seed, STREAM_ABSMAX, groups, 1.0)
    return Problem(packed=packed, scale_codes=codes, nested_absmax=absmax,
                   scale_codebook=scale_codebook(), value_codebook=nf4_style_codebook(),
                   offset=np.float32(offset), n=n, blocksize=blocksize, nested_blocksize=nbs)


def rotate_sets(problem: Problem, count: int):
    """Yield ``count`` independent copies of the problem's buffers (for L2 rotation)."""
    for _ in range(count):
        yield dataclasses.replace(problem, packed=problem.packed.copy(),
                                  scale_codes=problem.scale_codes.copy(),
                                  nested_absmax=problem.nested_absmax.copy())


def describe(problem: Problem, out: Optional[str] = None) -> str:
    npk, nb, ng = sizes(problem.n, problem.blocksize, problem.nested_blocksize)
    return (f"n={problem.n} bs={problem.blocksize} nbs={problem.nested_blocksize} "
            f"packed={npk}B codes={nb} absmax={ng} offset={float(problem.offset)!r}"
            + (f" out={out}" if out else ""))


# ------------------------------------------- LLM.int8 correction operands
STREAM_A = 11
STREAM_CB = 12
STREAM_SCB = 13
STREAM_COLS = 14


@dataclasses.dataclass
class Int8Problem:
    """Inputs of the LLM.int8 correction-operand preparation (host arrays)."""

    A_bits: np.ndarray  # uint16[M, K]: raw 16-bit activations (gathered bit for bit)
    CB: np.ndarray      # int8[N, K]: row-major int8 weights, the full code domain
    SCB: np.ndarray     # float32[N]: per-row statistics
    cols: np.ndarray    # int64[L]: outlier column indices in [0, K)

    @property
    def shape(self):
        return self.A_bits.shape[0], self.CB.shape[0], self.A_bits.shape[1], self.cols.size


def make_int8_problem(M: int, N: int, K: int, L: int, seed: int = 0,
                      cols_mode: str = "sorted", scb_sigma: float = 1.0) -> Int8Problem:
    """Random FP16-like activations, uniform int8 codes, lognormal row statistics.

    cols_mode: "sorted" (sorted distinct), "unsorted" (distinct, shuffled),
    "repeated" (with repeats), "edges" (contains 0 and K - 1).
    """
    a = uniform_bytes(seed, STREAM_A, 2 * M * K).view(np.uint16).reshape(M, K).copy()
    cb = uniform_bytes(seed, STREAM_CB, N * K).view(np.int8).reshape(N, K).copy()
    scb = lognormal_f32(seed, STREAM_SCB, N, scb_sigma)
    w = splitmix64(seed, STREAM_COLS, max(1, 4 * L))
    if L == 0:
        cols = np.zeros(0, dtype=np.int64)
    elif cols_mode == "repeated":
        cols = (w[:L] % np.uint64(K)).astype(np.int64)
        cols[L // 2:] = cols[:L - L // 2]
    else:
        # distinct columns: the L smallest random keys among a K-long key array
        keys = splitmix64(seed, STREAM_COLS + 100, K)
        pick = np.argsort(keys, kind="stable")[:L].astype(np.int64)
        if cols_mode == "sorted":
            cols = np.sort(pick)
        elif cols_mode == "edges":
            cols = np.sort(pick)
            cols[0], cols[-1] = 0, K - 1
        else:
            cols = pick
    return Int8Problem(A_bits=a, CB=cb, SCB=scb, cols=cols)


INT8_GRID_M = (1, 8, 64, 512, 2048)
INT8_GRID_KN = (3584, 4096, 8192, 14336)
INT8_GRID_L = (0, 1, 5, 16, 64)


# ------------------------------------------ dequantization feeding a GEMM
STREAM_G = 21


def make_integer_problem(rows: int, cols: int, blocksize: int = 64, nested_blocksize: int = 256,
                         seed: int = 0) -> Problem:
    """A nested problem whose dequantized values are small integers (|w| <= 16).

    Value codebook entries are integers in [-4, 3], scale codebook entries
    integers in [-4, 4], nested absmax 1 and offset 0, so every scale and
    every value is an exact integer.
    """
    p = make_problem(rows * cols, blocksize, nested_blocksize, "nf4", 0.5, 0.0, seed)
    vcb = (np.arange(16) % 8 - 4).astype(np.float32)
    scb = (np.arange(256) % 9 - 4).astype(np.float32)
    return dataclasses.replace(p, value_codebook=vcb, scale_codebook=scb,
                               nested_absmax=np.ones_like(p.nested_absmax),
                               offset=np.float32(0.0))


def make_ternary_g(rows: int, ncols: int, seed: int = 0) -> np.ndarray:
    """rows x ncols FP32 matrix of values in {-1, 0, 1}."""
    w = splitmix64(seed, STREAM_G, rows * ncols)
    return ((w % np.uint64(3)).astype(np.int64) - 1).astype(np.float32).reshape(rows, ncols)


def make_normal_g(rows: int, ncols: int, seed: int = 0) -> np.ndarray:
    """rows x ncols FP32 standard normal matrix (Box-Muller, float64, rounded once)."""
    return np.log(lognormal_f32(seed, STREAM_G, rows * ncols, 1.0).astype(np.float64)
                  ).astype(np.float32).reshape(rows, ncols)
