"""Pins for the CPU oracle of the 8-bit quantization (oracle/fp8.py).

The oracle's e4m3 encoder, its Walsh-Hadamard butterflies and its per-slice
scaling are tied to things other than themselves:
  * torch's float8_e4m3fn conversion (a library routine) and the format's
    definition (largest finite 448, subnormal step 2^-9, ties to even);
  * scipy's Sylvester-Hadamard matrix (a library routine) and H H^T = d I;
  * orthogonality of the rotation: rotated Q and K give the same Q K^T;
  * the round-trip bound of rounding to 3 mantissa bits;
  * planted mistakes, each of which must fail one of the pins.
"""
import math

import numpy as np
import pytest
import torch
from scipy.linalg import hadamard

import oracle.fp8 as of


def _signs(d, seed):
    return np.where(np.random.default_rng(seed).random(d) < 0.5, -1, 1).astype(np.int8)


def pin_encoder_matches_torch():
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(200000) * np.exp2(rng.integers(-14, 9, 200000))).astype(np.float32)
    v = np.concatenate([v, np.float32([0.0, -0.0, -2 ** -11, 2 ** -10, 3 * 2 ** -10, 1.5 * 2 ** -9, 2.5 * 2 ** -9,
                                       448, 464 - 1e-3, -448, 240, 248, 256, 272])])
    v = v[np.abs(v) < 464]  # torch's conversion does not saturate; beyond 464 it is NaN
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = of.e4m3_encode(v.astype(np.float64))
    assert np.array_equal(got, ref), int((got != ref).sum())


def pin_encoder_definition():
    assert of.e4m3_encode([448.0, 1e9, -1e9]).tolist() == [0x7E, 0x7E, 0xFE]   # saturation
    assert of.e4m3_encode([0.0, -0.0, -2.0 ** -11]).tolist() == [0x00, 0x80, 0x80]  # the sign of zero is kept
    assert of.e4m3_encode([2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10]).tolist() == [1, 0, 2]  # ties to even
    assert of.e4m3_encode([1.0, 1.0625, 1.1875]).tolist() == [0x38, 0x38, 0x3A]        # 1 + 1/16 ties down
    codes = np.arange(256, dtype=np.uint8)
    vals = of.e4m3_decode(codes)
    finite = ~np.isnan(vals)
    assert np.array_equal(of.e4m3_encode(vals[finite])[vals[finite] != 0], codes[finite][vals[finite] != 0])
    assert np.nanmax(vals) == 448.0 and np.isnan(vals[0x7F]) and np.isnan(vals[0xFF])


def pin_butterflies_match_hadamard_matrix():
    rng = np.random.default_rng(1)
    for d in (64, 128):
        s = _signs(d, d)
        x = rng.integers(-60, 60, (5, d)).astype(np.float32)  # sums stay exact in float32
        assert np.array_equal(of.hadamard_rows_f32(x, s).astype(np.float64), (x * s) @ hadamard(d))
        xf = rng.standard_normal((7, d)).astype(np.float32)
        np.testing.assert_allclose(of.hadamard_rows_f32(xf, s), (xf.astype(np.float64) * s) @ hadamard(d),
                                   rtol=1e-5, atol=1e-5)
        H = hadamard(d)
        assert np.array_equal(H @ H.T, d * np.eye(d))


def pin_rotation_is_orthogonal():
    rng = np.random.default_rng(2)
    d = 128
    s = _signs(d, 7)
    q = rng.standard_normal((1, 1, 9, d))
    k = rng.standard_normal((1, 1, 11, d))
    rq = of.hadamard_rows_f32(q, s).astype(np.float64) / math.sqrt(d)
    rk = of.hadamard_rows_f32(k, s).astype(np.float64) / math.sqrt(d)
    np.testing.assert_allclose(rq[0, 0] @ rk[0, 0].T, q[0, 0] @ k[0, 0].T, rtol=1e-4, atol=1e-4)


def pin_quantize_round_trip():
    rng = np.random.default_rng(3)
    for rotate in (False, True):
        for d in (64, 128):
            x = (rng.standard_normal((2, 3, 50, d)) * np.exp2(rng.integers(-3, 4, (2, 3, 1, 1)))).astype(np.float32)
            s = _signs(d, 11) if rotate else None
            codes, desc = of.fp8_quantize(x, s)
            y = of.hadamard_rows_f32(x, s).astype(np.float64) / math.sqrt(d) if rotate else x.astype(np.float64)
            back = of.fp8_dequantize(codes, desc)
            # Each value is rounded to 3 mantissa bits (half-ulp 2^-4 relative) or, below
            # 2^-6 of the scaled range, to a multiple of 2^-9 (half-step 2^-10).
            step = np.maximum(2.0 ** -4 * np.abs(y), 2.0 ** -10 * desc[:, :, None, None])
            assert np.all(np.abs(back - y) <= step * (1 + 1e-6)), (rotate, d)
            # The slice maximum lands exactly on +-448.
            for b in range(2):
                for h in range(3):
                    i = np.argmax(np.abs(y[b, h]))
                    assert int(codes[b, h].reshape(-1)[i]) & 0x7F == 0x7E
            ct, dt = of.fp8_quantize(x, s, transpose=True)
            assert np.array_equal(ct, np.swapaxes(codes, 2, 3)) and np.array_equal(dt, desc)


def pin_zero_slice():
    x = np.zeros((1, 2, 16, 64), dtype=np.float32)
    x[0, 1, 3, 5] = 2.0
    codes, desc = of.fp8_quantize(x, _signs(64, 1))
    assert not codes[0, 0].any() and desc[0, 0] == 0.0
    assert desc[0, 1] > 0.0


PINS = [("encoder_torch", pin_encoder_matches_torch), ("encoder_definition", pin_encoder_definition),
        ("butterflies", pin_butterflies_match_hadamard_matrix), ("orthogonal", pin_rotation_is_orthogonal),
        ("round_trip", pin_quantize_round_trip), ("zero_slice", pin_zero_slice)]


@pytest.mark.parametrize("name,check", PINS, ids=[n for n, _ in PINS])
def test_oracle_fp8_pin(name, check):
    check()


# --------------------------------------------------------------------------
# Planted mistakes: each must fail at least one pin.
# --------------------------------------------------------------------------

def _bad_butterflies(kind):
    good = of.hadamard_rows_f32

    def f(x, signs):
        if kind == "no_signs":
            return good(x, np.ones_like(np.asarray(signs)))
        if kind == "upper_plus":
            y = np.asarray(x, dtype=np.float32) * np.asarray(signs, dtype=np.float32)
            d = y.shape[-1]
            h = 1
            while h < d:
                z = y.reshape(y.shape[:-1] + (d // (2 * h), 2, h))
                a, b = z[..., 0, :].copy(), z[..., 1, :].copy()
                z[..., 0, :] = a + b
                z[..., 1, :] = b - a
                y = z.reshape(y.shape)
                h *= 2
            return y
        if kind == "stop_early":
            return good(x, signs) if x.shape[-1] < 4 else _partial(x, signs)
        raise ValueError(kind)

    def _partial(x, signs):
        y = np.asarray(x, dtype=np.float32) * np.asarray(signs, dtype=np.float32)
        d = y.shape[-1]
        h = 1
        while h < d // 2:
            z = y.reshape(y.shape[:-1] + (d // (2 * h), 2, h))
            a, b = z[..., 0, :].copy(), z[..., 1, :].copy()
            z[..., 0, :] = a + b
            z[..., 1, :] = a - b
            y = z.reshape(y.shape)
            h *= 2
        return y
    return f


def _run_pins():
    failures = 0
    for _, check in PINS:
        try:
            check()
        except (AssertionError, ValueError, IndexError):
            failures += 1
    return failures


@pytest.mark.parametrize("kind", ["no_signs", "upper_plus", "stop_early"])
def test_planted_rotation_mistakes_are_caught(kind, monkeypatch):
    monkeypatch.setattr(of, "hadamard_rows_f32", _bad_butterflies(kind))
    assert _run_pins() > 0


def test_planted_scaling_mistakes_are_caught(monkeypatch):
    good = of.fp8_quantize

    def no_sqrt(x, signs=None, transpose=False):
        codes, desc = good(x, signs, transpose)
        return codes, desc * np.float32(math.sqrt(x.shape[-1]) if signs is not None else 1.0)
    monkeypatch.setattr(of, "fp8_quantize", no_sqrt)
    assert _run_pins() > 0


def test_planted_rounding_mistake_is_caught(monkeypatch):
    good = of.e4m3_encode
    monkeypatch.setattr(of, "e4m3_encode", lambda x: good(np.asarray(x, dtype=np.float64) * (1 + 2.0 ** -6)))
    assert _run_pins() > 0
