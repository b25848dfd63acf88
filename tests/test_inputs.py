"""The seeded input generator (no attention arithmetic lives there)."""
import numpy as np
import pytest

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


# --------------------------------------------------------------------------
# e4m3 codec used for the 8-bit path's inputs
# --------------------------------------------------------------------------

def test_e4m3_decode_spot_values():
    """Values fixed by the E4M3 format (1 sign, 4 exponent bits with bias 7,
    3 mantissa bits; S.1111.111 is NaN; no infinities)."""
    from fa_inputs import e4m3_bits_to_f64
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x39: 1.125,
             0x40: 2.0, 0x77: 240.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0, 0x80: -0.0}
    for code, val in cases.items():
        assert e4m3_bits_to_f64(np.array([code], dtype=np.uint8))[0] == val, hex(code)
    assert np.isnan(e4m3_bits_to_f64(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_e4m3_encode_round_trip_and_rounding():
    from fa_inputs import e4m3_bits_to_f64, f64_to_e4m3_bits
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF, 0x80)], dtype=np.uint8)
    assert np.array_equal(f64_to_e4m3_bits(e4m3_bits_to_f64(codes)), codes)
    # ties go to the even code; saturation at 448
    x = np.array([2.0 ** -10, 1.5 * 2.0 ** -9, 1.0625, 1.1875, 449.0, 1e6, -1e6])
    want = np.array([0x00, 0x02, 0x38, 0x3A, 0x7E, 0x7E, 0xFE], dtype=np.uint8)
    assert np.array_equal(f64_to_e4m3_bits(x), want)
    # monotone, and within half an ulp of the input in range
    rng = np.random.default_rng(3)
    x = np.sort(rng.uniform(-448, 448, 5000))
    y = e4m3_bits_to_f64(f64_to_e4m3_bits(x))
    assert np.all(np.diff(y) >= 0)
    big = np.abs(x) >= 2.0 ** -6
    assert np.all(np.abs(y - x)[big] <= np.abs(x)[big] * 2.0 ** -4 + 1e-12)


def test_e4m3_matches_torch_float8():
    """torch's float8_e4m3fn conversion (a library routine) agrees inside the range."""
    import torch
    from fa_inputs import f64_to_e4m3_bits
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.standard_normal(4000) * s for s in (1e-3, 0.1, 1.0, 30.0)])
    x = np.clip(x, -448, 448).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(f64_to_e4m3_bits(x.astype(np.float64)), ref)


def test_fp8_problem_scales():
    from fa_inputs import make_dense, make_fp8, bf16_bits_to_f64
    p = make_dense(2, 4, 2, 40, 48, 128, seed=9, causal=True)
    f = make_fp8(p)
    assert f.vt8.shape == (2, 2, 128, 48) and f.q_scale.shape == (2, 4)
    q, k, v = f.dequantized()
    for x, ref in ((q, p.q), (k, p.k), (v, p.v)):
        r = bf16_bits_to_f64(ref)
        amax = np.abs(r).max(axis=(2, 3), keepdims=True)
        assert np.all(np.abs(x - r) <= amax * 2.0 ** -4 + 1e-12)   # half an ulp at the slice's scale
        assert np.allclose(np.abs(x).max(axis=(2, 3)), amax[..., 0, 0], rtol=2.0 ** -4)
