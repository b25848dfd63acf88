"""CPU oracle for the 8-bit path's quantization (block scaling and incoherent processing).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module;
only the tests and the smoke check may call it.

The FA3 canvas ("FlashAttention v3 Hopper asynchrony: TMA + WGMMA + ping-pong",
element ``pseudo-code``) lists block scaling of Q/K/V and incoherent processing
for its FP8 path, and the interview canvas ("FlashAttention面试讲解", element
``script-body``) says both keep the low-precision path accurate.  Neither
defines them.  The readings used here:

* block = one (batch, head) slice of a tensor; scale = 448 / max |value| over
  the slice, so the slice's largest value maps to e4m3's largest finite 448;
* incoherent processing = every row times M = diag(signs) H_d / sqrt(d), with
  H_d the Sylvester-Hadamard matrix (H[i, j] = (-1)^popcount(i & j)) and
  signs a random +-1 vector; M is orthogonal, so Q M (K M)^T = Q K^T.

Since the quantized value is an integer code, the decision is taken in the
precision the kernel uses (float32).  (x * signs) H_d is formed by the
Walsh-Hadamard butterflies with strides 1, 2, ..., d/2, so that float32 sums
happen in one fixed order.  Then inv = 448 / max|y| (float32),
code = e4m3(y * inv) and descale = max|y| / (448 sqrt(d)) (or / 448 unrotated,
float64 then float32).  e4m3 is the OCP 8-bit format E4M3: 1 sign, 4 exponent
(bias 7) and 3 mantissa bits, no infinities, largest finite 448, subnormals
m * 2^-9.  Rounding is to nearest with ties to the even mantissa, saturating
at +-448; the sign bit is copied from the input, so -0.0 encodes as 0x80.

Pins: ``tests/test_oracle_fp8.py`` (the Hadamard matrix of scipy, torch's
float8_e4m3fn conversion, orthogonality, round-trip bounds, planted mistakes).
"""
from __future__ import annotations

import math
from typing import Optional, Tuple

import numpy as np

E4M3_LARGEST = 448.0


def e4m3_encode(x) -> np.ndarray:
    """e4m3 codes (uint8) of finite values: nearest value, ties to the even
    mantissa, saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    code = np.zeros(x.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    # Subnormal range: multiples of 2^-9 (m = 8 rounds up to 2^-6, code 8).
    code = np.where(sub, np.rint(a * 2.0 ** 9), code)
    # Normal range: a = (m8 / 8) * 2^e with m8 in [8, 16).
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(sub, 1.0, a)))
    m8 = np.rint(np.where(sub, 8.0, a) / np.exp2(e - 3))
    carry = m8 >= 16
    e = np.where(carry, e + 1, e)
    m8 = np.where(carry, 8, m8)
    normal_code = (e + 7) * 8 + (m8 - 8)
    code = np.where(sub, code, normal_code)
    code = np.minimum(code, 0x7E)  # saturate at 448 (0x7F is NaN)
    code = code.astype(np.uint8)
    # The sign bit is the input's, zero included (-0.0 encodes as 0x80).
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    """Values (float64) of e4m3 codes; NaN for the NaN codes."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    mag = c & 0x7F
    e = mag >> 3
    m = mag & 7
    val = np.where(e == 0, m * 2.0 ** -9, (8 + m) * np.exp2(e.astype(np.float64) - 10))
    val = np.where(mag == 0x7F, np.nan, val)
    return np.where(c & 0x80, -val, val)


def hadamard_rows_f32(x, signs) -> np.ndarray:
    """(x * signs) H_d along the last axis, in float32 by the radix-2
    Walsh-Hadamard butterflies (stride h pairs i and i + h, i & h == 0:
    lower <- a + b, upper <- a - b), strides 1, 2, 4, ..., d/2."""
    y = np.asarray(x, dtype=np.float32) * np.asarray(signs, dtype=np.float32)
    d = y.shape[-1]
    assert d & (d - 1) == 0, "d must be a power of two"
    h = 1
    while h < d:
        z = y.reshape(y.shape[:-1] + (d // (2 * h), 2, h))
        a = z[..., 0, :].copy()
        b = z[..., 1, :].copy()
        z[..., 0, :] = a + b
        z[..., 1, :] = a - b
        y = z.reshape(y.shape)
        h *= 2
    return y


def fp8_quantize(x, signs: Optional[np.ndarray] = None, transpose: bool = False) -> Tuple[np.ndarray, np.ndarray]:
    """Codes and per-(batch, head) descales of x [B, H, N, d] (float values,
    e.g. bf16 inputs widened).  Returns (codes [B, H, N, d] or, transposed,
    [B, H, d, N] uint8; descale [B, H] float32)."""
    x = np.asarray(x, dtype=np.float32)
    B, H, N, d = x.shape
    y = hadamard_rows_f32(x, signs) if signs is not None else x
    amax = np.abs(y).max(axis=(2, 3)) if N > 0 else np.zeros((B, H), dtype=np.float32)
    amax = amax.astype(np.float32)
    inv = np.where(amax > 0, np.float32(448.0) / np.where(amax > 0, amax, np.float32(1.0)), np.float32(0.0))
    inv = inv.astype(np.float32)
    scaled = (y * inv[:, :, None, None]).astype(np.float32)
    codes = e4m3_encode(scaled.astype(np.float64))
    divisor = 448.0 * (math.sqrt(d) if signs is not None else 1.0)
    descale = (amax.astype(np.float64) / divisor).astype(np.float32)
    if transpose:
        codes = np.ascontiguousarray(np.swapaxes(codes, 2, 3))
    return codes, descale


def fp8_dequantize(codes, descale, transpose: bool = False) -> np.ndarray:
    """codes * descale in float64, back in the [B, H, N, d] layout."""
    v = e4m3_decode(codes) * np.asarray(descale, dtype=np.float64)[:, :, None, None]
    return np.swapaxes(v, 2, 3) if transpose else v
