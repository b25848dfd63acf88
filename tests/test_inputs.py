"""The seeded input generator (no attention arithmetic lives there)."""
import numpy as np

from fa_inputs import (raw_u64, normal_f32, f32_to_bf16_bits, bf16_bits_to_f32, make_dense,
                       make_varlen, varlen_lengths, scale_outliers_bf16, stream_key, WORKLOADS,
                       make_workload)


def test_splitmix64_published_sequence():
    # SplitMix64 started from state 0 (Vigna's reference splitmix64.c).
    got = [int(x) for x in raw_u64(0, 0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_streams_are_random_access():
    a = raw_u64(12345, 0, 100)
    b = raw_u64(12345, 40, 10)
    assert np.array_equal(a[40:50], b)


def test_normal_moments():
    z = normal_f32(stream_key(3, 1), 1 << 20)
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1.0) < 5e-3


def test_bf16_rounding_ties_to_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -7], dtype=np.float32)
    back = bf16_bits_to_f32(f32_to_bf16_bits(x))
    assert back.tolist() == [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 1.0 + 2 ** -7]


def test_outliers_exact_and_fraction():
    k = make_dense(1, 1, 1, 1, 4096, 128, seed=4, causal=True).k
    k2 = scale_outliers_bf16(k, stream_key(4, 4), 0.01, 8)
    a, b = bf16_bits_to_f32(k), bf16_bits_to_f32(k2)
    changed = a != b
    assert 0.008 < changed.mean() < 0.012
    assert np.array_equal(b[changed], a[changed] * 8)


def test_workload_shapes():
    p = make_dense(2, 4, 2, 10, 12, 64, seed=1, causal=True)
    assert p.q.shape == (2, 4, 10, 64) and p.k.shape == (2, 2, 12, 64)
    lens = varlen_lengths(5)
    assert len(lens) == 16 and all(256 <= x <= 8192 for x in lens)
    pv = make_varlen([3, 0, 5], 2, 1, 64, seed=2, causal=True)
    assert pv.q.shape == (2, 8, 64) and list(pv.cu_seqlens) == [0, 3, 3, 8] and pv.Nq == 5
    t = make_workload("tiny_b1_h2_n128_d64")
    assert t.q.shape == (1, 2, 128, 64) and abs(t.flops() - 8.388608e6) < 1
    assert set(WORKLOADS) >= {"b2_h32_n4096_d128_causal", "varlen16_h16_d128_causal"}
