"""The seeded synthetic input generators (no attention arithmetic)."""
import numpy as np

import alibi_inputs as gen


def test_splitmix64_reference_values():
    # SplitMix64 from state 0: the first two outputs of the published generator.
    G = gen.GOLDEN
    assert int(gen.mix64(np.array([G], dtype=np.uint64))[0]) == 0xE220A8397B1DCDAF
    assert int(gen.mix64(np.array([(2 * G) % (1 << 64)], dtype=np.uint64))[0]) == 0x6E789E6AA1B965F4


def test_c_stream_matches_numpy_stream():
    # uniform(-1, 1) = -1 + 2 u01 with u01 = (u64 >> 11) 2^-53: the C core and the
    # numpy integer stream must agree bit for bit.
    for seed, sid, start in [(42, 0, 0), (42, 2, 123456), (7, 5, 10 ** 9)]:
        u64 = gen.counter_u64(seed, sid, start, 5000)
        want = (-1.0 + 2.0 * ((u64 >> np.uint64(11)).astype(np.float64) * 2.0 ** -53)).astype(np.float32)
        got = gen.uniform(seed, sid, 5000, -1.0, 1.0, start=start)
        assert np.array_equal(got, want)


def test_counter_generator_is_deterministic_and_sliceable():
    a = gen.normal(42, 3, 300_000)
    b = gen.normal(42, 3, 100_000, start=200_000)
    assert np.array_equal(a[200_000:], b)
    assert np.array_equal(a, gen.normal(42, 3, 300_000, nthreads=1))
    assert not np.array_equal(a, gen.normal(42, 4, 300_000))
    assert not np.array_equal(a, gen.normal(43, 3, 300_000))


def test_normal_and_uniform_moments():
    x = gen.normal(42, 0, 1_000_000).astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1.0) < 5e-3
    assert abs(np.mean(x ** 4) - 3.0) < 0.05  # Gaussian kurtosis
    u = gen.uniform(42, 2, 1_000_000, -1.0, 1.0).astype(np.float64)
    assert u.min() >= -1.0 and u.max() < 1.0 and abs(u.mean()) < 5e-3
    assert abs(u.var() - 1.0 / 3.0) < 5e-3


def test_bf16_rounding_ties_to_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 0.0], np.float32)
    back = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(vals))
    # 1 + 2^-8 ties between 1 and 1 + 2^-7 -> even (1.0); 1 + 3 2^-8 ties -> 1 + 2^-6
    assert list(back) == [1.0, 1.0, 1.0 + 2 ** -6, 1.0, -2.5, 0.0]


def test_workload_shapes_and_slices():
    q, k, v = gen.generate(gen.WORKLOADS["tiny_fp32"])
    assert q.shape == (1, 4, 64, 16) and q.bf16 is None and q.f32.dtype == np.float32
    st = np.random.RandomState(42)
    assert np.array_equal(q.f32, (st.randn(1, 4, 64, 16) * 0.5).astype(np.float32))
    w = gen.WORKLOADS["heads6_n1024"].with_n(100)
    q, k, v = gen.generate(w)
    assert q.shape == (2, 6, 100, 64) and q.bf16.dtype == np.uint16
    assert np.array_equal(gen.bf16_bits_to_f32(q.bf16), q.f32)
    hs = gen.head_slice(w, 1, 1, 4)
    assert np.array_equal(hs.bf16, k.bf16[1, 4])
    wd = gen.WORKLOADS["decode_l8192"]
    qs, ks, vs = wd.shapes()
    assert qs == (64, 40, 128) and ks == (64, 40, 8192, 128)
