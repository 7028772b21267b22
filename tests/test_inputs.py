"""The seeded synthetic input generators (no attention arithmetic)."""
import numpy as np

import alibi_inputs as gen


def test_counter_generator_is_deterministic_and_sliceable():
    a = gen.counter_u64(42, 3, 0, 1000)
    b = gen.counter_u64(42, 3, 500, 500)
    assert np.array_equal(a[500:], b)
    assert not np.array_equal(a, gen.counter_u64(42, 4, 0, 1000))
    assert not np.array_equal(a, gen.counter_u64(43, 3, 0, 1000))


def test_splitmix64_reference_values():
    # SplitMix64 with state 0: the first outputs of the published generator.
    z = np.array([0x9E3779B97F4A7C15], dtype=np.uint64)
    assert int(gen._mix64(z)[0]) == 0xE220A8397B1DCDAF
    z2 = np.array([(2 * 0x9E3779B97F4A7C15) % (1 << 64)], dtype=np.uint64)
    assert int(gen._mix64(z2)[0]) == 0x6E789E6AA1B965F4


def test_normal_and_uniform_moments():
    x = gen.counter_normal(42, 0, 400_000)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    u = gen.counter_uniform(42, 2, 400_000, -1.0, 1.0)
    assert u.min() >= -1.0 and u.max() < 1.0 and abs(u.mean()) < 0.01
    assert abs(u.var() - 1.0 / 3.0) < 0.01


def test_bf16_rounding_ties_to_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 0.0], np.float32)
    bits = gen.f32_to_bf16_bits(vals)
    back = gen.bf16_bits_to_f32(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa -> 1.0
    # 1 + 3*2^-8 is a tie between 1 + 2^-7 and 1 + 2^-6: even -> 1 + 2^-6
    assert list(back) == [1.0, 1.0, 1.0 + 2 ** -6, 1.0, -2.5, 0.0]


def test_workload_shapes_and_dtypes():
    q, k, v = gen.generate(gen.WORKLOADS["tiny_fp32"])
    assert q.shape == (1, 4, 64, 16) and q.bf16 is None and q.f32.dtype == np.float32
    # tiny workload follows the legacy MT19937 seed-42 recipe
    st = np.random.RandomState(42)
    assert np.array_equal(q.f32, (st.randn(1, 4, 64, 16) * 0.5).astype(np.float32))
    q, k, v = gen.generate(gen.WORKLOADS["heads6_n1024"], scale_n=100)
    assert q.shape == (2, 6, 100, 64) and q.bf16.dtype == np.uint16
    assert np.array_equal(gen.bf16_bits_to_f32(q.bf16), q.f32)
    w = gen.WORKLOADS["decode_l8192"]
    qs, ks, vs = w.shapes()
    assert qs == (64, 40, 128) and ks == (64, 40, 8192, 128)
