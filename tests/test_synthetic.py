"""The seeded input generator (CPU only)."""
import numpy as np

import synthetic as syn


def test_deterministic_and_sliceable():
    a = syn.normal_bf16(7, 2, (1000,))
    b = syn.normal_bf16(7, 2, (1000,))
    assert np.array_equal(a, b)
    # any sub-range regenerates to the same values, odd starts included
    for first, n in [(0, 10), (1, 9), (333, 100), (999, 1)]:
        assert np.array_equal(syn.normal_bf16(7, 2, (n,), first=first), a[first:first + n])
    assert not np.array_equal(a, syn.normal_bf16(8, 2, (1000,)))
    assert not np.array_equal(a, syn.normal_bf16(7, 3, (1000,)))


def test_normal_moments():
    x = syn.bf16_bits_to_f32(syn.normal_bf16(1, 1, (200000,))).astype(np.float64)
    assert abs(x.mean()) < 0.01
    assert abs(x.var() - 1) < 0.02
    assert abs((x ** 4).mean() - 3) < 0.1   # normal kurtosis
    assert np.all(np.isfinite(x))


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e38, 1e-40], dtype=np.float32)
    bits = syn.f32_to_bf16_bits(vals)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa (1.0) wins
    assert bits[1] == 0x3F80
    # 1 + 3*2^-8 is a tie between 1+2^-7 and 1+2^-6: even mantissa wins
    assert bits[2] == 0x3F82
    back = syn.bf16_bits_to_f32(bits)
    assert back[0] == 1.0 and back[3] == -2.5


def test_uniform_int_range():
    x = syn.uniform_int(3, 4, 100000, 512, 32768)
    assert x.min() >= 512 and x.max() <= 32768
    assert abs(x.mean() - (512 + 32768) / 2) < 200
    y = syn.uniform_int(3, 4, 100000, 5, 5)
    assert np.all(y == 5)


def test_fill_cache_layout_and_tail():
    B, G, Tmax, D = 3, 2, 10, 4
    lens = np.array([10, 3, 0], dtype=np.int32)
    c = syn.fill_cache(5, 2, B, G, Tmax, D, lens, syn.BF16_NAN, threads=2)
    for b in range(B):
        for g in range(G):
            T = lens[b]
            assert np.array_equal(c[b, g, :T], syn.cache_slice(5, 2, G, Tmax, D, b, g, T))
            assert np.all(c[b, g, T:] == syn.BF16_NAN)
    one = syn.fill_cache(5, 2, B, G, Tmax, D, lens, syn.BF16_NAN, threads=1)
    assert np.array_equal(c, one)


def test_ragged_lengths_of_the_ragged_workload():
    cfg = syn.config_by_name("ragged_sq4")
    lens = syn.seq_lens_for(cfg)
    assert lens.shape == (64,) and lens.min() >= 512 and lens.max() <= 32768
    assert np.array_equal(lens, syn.seq_lens_for(cfg))
