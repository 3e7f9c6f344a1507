"""The seeded input generator: determinism, distributions, bfloat16 rounding."""
import numpy as np

import gen


def test_counter_based_and_deterministic():
    a = gen.words(0, 1, 0, 1000)
    b = gen.words(0, 1, 0, 1000)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(gen.words(0, 1, 400, 100), a[400:500])
    assert not np.array_equal(gen.words(0, 2, 0, 1000), a)
    assert not np.array_equal(gen.words(1, 1, 0, 1000), a)
    # any window of a tensor equals the same window of a longer draw
    z = gen.normals_f64(5, 0, 1001)
    np.testing.assert_array_equal(gen.normals_f64(5, 0, 10, start=333), z[333:343])


def test_splitmix64_reference_values():
    # SplitMix64 with state 0: the first outputs of the published generator
    # (Steele, Lea & Flood 2014; same constants as java.util.SplittableRandom).
    g = np.uint64(0x9E3779B97F4A7C15)
    with np.errstate(over="ignore"):
        n = np.arange(1, 4, dtype=np.uint64) * g
    got = gen._mix64(n)
    expect = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert [int(x) for x in got] == expect


def test_normal_moments():
    z = gen.normals_f64(0, 0, 400_000)
    assert abs(z.mean()) < 0.01
    assert abs(z.std() - 1.0) < 0.01
    assert abs(np.mean(z ** 4) - 3.0) < 0.05


def test_bf16_rounding_is_nearest_even():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 4.0,
                        # exact ties between two bfloat16 neighbours
                        (np.arange(1, 200) * 2 + 1) * 2.0 ** -8 + 1.0, [0.0, -0.0]])
    bits = gen.f64_to_bf16_bits(x)
    got = gen.bf16_bits_to_f64(bits)
    for xi, gi, bi in zip(x, got, bits):
        if xi == 0:
            assert gi == 0
            continue
        e = np.floor(np.log2(abs(xi)))
        ulp = 2.0 ** (e - 7)
        lo = np.floor(xi / ulp) * ulp
        hi = lo + ulp
        if abs(xi - lo) < abs(hi - xi):
            want = lo
        elif abs(xi - lo) > abs(hi - xi):
            want = hi
        else:  # tie: even significand
            want = lo if int(round(lo / ulp)) % 2 == 0 else hi
        assert gi == want, (xi, gi, want)


def test_lengths_uniform_inclusive():
    L = gen.lengths(0, 20000, 8, 64)
    assert L.min() == 8 and L.max() == 64
    counts = np.bincount(L - 8, minlength=57)
    assert counts.min() > 250 and counts.max() < 460  # 351 expected per value
    np.testing.assert_array_equal(gen.lengths(0, 256, 8, 64), L[:256])


def test_workload_shapes():
    spec = gen.WORKLOADS["cross_pad_bf16_b64_h16_lq96_lk128_d64"]
    small = dict(spec, B=2, H=2)
    q, k, v, lens = gen.make_inputs(small)
    assert q.shape == (2, 2, 96, 64) and q.dtype == np.uint16
    assert k.shape == (2, 2, 128, 64) and v.shape == (2, 2, 128, 64)
    assert lens.shape == (2,) and np.all((lens >= 16) & (lens <= 128))
    assert gen.default_scale(64) == 0.125
    assert gen.default_scale(128) == float(np.float32(1 / np.sqrt(128.0)))
