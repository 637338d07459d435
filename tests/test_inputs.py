"""The seeded generator: deterministic, the right sizes, and the stated distributions."""

import numpy as np

import dq4_inputs as gen


def test_splitmix64_known_values():
    # splitmix64 from state 0 (Steele/Lea/Flood; also Vigna's reference C code):
    # the first outputs for seed state 0 are fixed numbers.
    z = np.array([0], dtype=np.uint64)
    with np.errstate(over="ignore"):
        w = gen._mix(z + np.arange(1, 4, dtype=np.uint64) * gen.GOLDEN)
    assert [int(x) for x in w] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_stream_separated():
    a = gen.make_problem(10_001, 64, 256, "nf4", 0.5, 0.1, seed=3)
    b = gen.make_problem(10_001, 64, 256, "nf4", 0.5, 0.1, seed=3)
    c = gen.make_problem(10_001, 64, 256, "nf4", 0.5, 0.1, seed=4)
    assert np.array_equal(a.packed, b.packed) and np.array_equal(a.nested_absmax, b.nested_absmax)
    assert not np.array_equal(a.packed, c.packed)
    assert not np.array_equal(a.packed[:157], a.scale_codes[:157])


def test_sizes_match_cells():
    c1 = gen.CELLS["C1"].problem()
    assert c1.packed.size == 8_388_608 and c1.scale_codes.size == 262_144
    assert c1.nested_absmax.size == 1_024
    assert gen.CELLS["C1"].algorithmic_bytes() == 42_210_368
    assert gen.CELLS["C4a"].algorithmic_bytes() == 590_931_008
    npk, nb, ng = gen.sizes(4097 * 4095, 64, 256)
    assert (npk, nb, ng) == (8_388_608, 262_144, 1_024)


def test_codebooks():
    scb = gen.scale_codebook()
    assert scb.dtype == np.float32 and scb.size == 256
    assert scb[0] == -1 and scb[-1] == 1 and np.all(np.diff(scb) > 0)
    assert np.array_equal(scb, -scb[::-1])
    for name, cb in (("nf4", gen.nf4_style_codebook()), ("fp4", gen.fp4_style_codebook())):
        assert cb.dtype == np.float32 and cb.size == 16, name
        assert cb[0] == -1 and cb[-1] == 1 and 0.0 in cb, name
        assert np.all(np.diff(cb) >= 0), name
    fp4 = gen.fp4_style_codebook()
    assert np.signbit(fp4[7]) and fp4[7] == 0 and not np.signbit(fp4[8])


def test_lognormal_statistics():
    x = gen.lognormal_f32(1, gen.STREAM_ABSMAX, 200_000, 0.5)
    z = np.log(x.astype(np.float64))
    assert abs(z.mean()) < 0.01 and abs(z.std() - 0.5) < 0.01
    assert np.all(x > 0)


def test_uniform_codes():
    p = gen.CELLS["C1"].problem()
    counts = np.bincount(p.scale_codes, minlength=256)
    assert counts.min() > 0.8 * counts.mean()
    nib = np.concatenate([p.packed >> 4, p.packed & 15])
    c16 = np.bincount(nib, minlength=16)
    assert c16.min() > 0.95 * c16.mean()


def test_force_all_codes():
    p = gen.make_problem(64 * 300 + 17, 64, 256, "fp4", 0.5, 1.0, seed=9, force_all_codes=True)
    assert np.array_equal(p.scale_codes[:256], np.arange(256))
    for b in range(p.nblocks - 1):
        bytes_ = p.packed[b * 32:b * 32 + 8]
        nib = np.stack([bytes_ >> 4, bytes_ & 15], axis=1).ravel()
        assert np.array_equal(nib, np.arange(16))


def test_enumeration_problem_covers_grid():
    p = gen.enumeration_problem(0.52)
    nib = np.stack([p.packed >> 4, p.packed & 15], axis=1).ravel()
    seen = {(b // 256, int(p.scale_codes[b]), int(k)) for b in range(p.nblocks)
            for k in set(nib[b * 32:(b + 1) * 32].tolist())}
    assert len(seen) == 4 * 256 * 16
