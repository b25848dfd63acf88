"""GPU parity of fa_fp8_quantize (block scaling and incoherent processing for
the 8-bit path) against the CPU oracle in oracle/fp8.py, and of the 8-bit
forward fed by it.

The quantized codes are integers decided in float32 on both sides (the
Walsh-Hadamard butterflies in one fixed order, 448 / max|y| correctly
rounded, one float32 product, round to nearest even), so they must match bit
for bit, and so must the descales.  The forward on quantized inputs is then
held to the 8-bit bound of the forward's own tests (P rounded to e4m3):

    |O_gpu - O_ref| <= 2^-4 * attention(|V|) + 2^-8 |O_ref| + 2e-3,

with the oracle run on the dequantized (rotated) Q and K and dequantized V.
Finally the point of the rotation: with a few large channels in Q and K, it
must lower the error against the exact bf16 attention.
"""
import math

import numpy as np
import pytest
import torch

from fa_inputs import (bf16_bits_to_f32, bf16_bits_to_f64, f64_to_bf16_bits, make_dense, normal_bf16,
                       scale_outliers_bf16, stream_key)
from oracle import attention_fwd
from oracle.fp8 import fp8_dequantize, fp8_quantize

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_42_gb300 as m
    m.build()
    m.lib()
    return m


@pytest.fixture(scope="module")
def dev():
    return torch.device("cuda", 0)


@pytest.fixture(autouse=True)
def _status_clean(fa):
    fa.fa_device_status()
    yield
    assert fa.fa_device_status() == 0, "a kernel wait timed out"


def _to_dev(bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


CASES = [
    # (B, H, N, d, rotate, transpose, outliers)
    (1, 2, 128, 128, True, False, False),
    (2, 3, 200, 128, False, False, False),   # ragged last block of rows
    (1, 2, 336, 64, True, False, True),      # d = 64, entries scaled by 2^6
    (2, 2, 208, 128, True, True, False),     # transposed, 208 = 3 blocks + 16 rows
    (1, 3, 64, 64, False, True, True),
    (1, 1, 1000, 128, True, False, True),    # many blocks per slice
    # The one-launch path takes slices of up to 1024 rows (above) and plain
    # slices up to its shared-memory limit (a 16-CTA cluster per slice) ...
    (2, 2, 4096, 128, False, False, True),
    (1, 1, 8192, 64, False, False, False),
    # ... the four-launch path large rotated or transposed slices, and slices
    # past that limit.
    (1, 2, 4096, 128, False, True, False),
    (1, 1, 8192, 64, True, False, True),
    (1, 2, 4160, 128, False, False, False),
    (1, 1, 8208, 64, False, True, False),
    (1, 2, 4096, 128, True, False, True),    # rotated d = 128, four launches
    (2, 1, 2048, 128, True, True, False),    # rotated and transposed
    # Tensors near or above the L2 size (the GQA N16384 inputs).
    (1, 32, 16384, 128, False, True, False),  # 134 MB, transposed
    (1, 26, 16384, 128, True, False, False),  # 109 MB, rotated
]


@pytest.mark.parametrize("B,H,N,d,rotate,transpose,outliers", CASES)
def test_codes_and_descales_match_the_oracle(fa, dev, B, H, N, d, rotate, transpose, outliers):
    seed = 100 + B * 7 + H * 5 + N + d
    bits = normal_bf16(stream_key(seed, 1), (B, H, N, d))
    if outliers:
        bits = scale_outliers_bf16(bits, stream_key(seed, 2), 0.002, 64)
    if B * H > 1:
        bits[-1, -1] = 0  # an all-zero slice
    signs = fa.hadamard_signs(d, seed, dev) if rotate else None
    x8, desc = fa.fp8_quantize(_to_dev(bits, dev), signs, transpose=transpose)
    torch.cuda.synchronize(dev)
    ref8, ref_desc = fp8_quantize(bf16_bits_to_f32(bits), None if signs is None else signs.cpu().numpy(),
                                  transpose=transpose)
    got8 = x8.cpu().numpy()
    assert got8.shape == ref8.shape
    bad = got8 != ref8
    assert not bad.any(), "%d codes differ, first at %s" % (bad.sum(), np.argwhere(bad)[0])
    assert np.array_equal(desc.cpu().numpy(), ref_desc)


def test_empty_rows_give_zero_descales(fa, dev):
    x = torch.zeros((2, 3, 0, 128), dtype=torch.bfloat16, device=dev)
    x8, desc = fa.fp8_quantize(x, fa.hadamard_signs(128, 1, dev), transpose=True)
    torch.cuda.synchronize(dev)
    assert x8.shape == (2, 3, 128, 0) and torch.all(desc == 0)


def test_rotated_quantized_forward_parity(fa, dev):
    p = make_dense(1, 4, 2, 200, 256, 128, seed=31, causal=True)
    signs = fa.hadamard_signs(128, 9, dev)
    q8, qd = fa.fp8_quantize(_to_dev(p.q, dev), signs)
    k8, kd = fa.fp8_quantize(_to_dev(p.k, dev), signs)
    vt8, vd = fa.fp8_quantize(_to_dev(p.v, dev), None, transpose=True)
    o, lse = fa.fwd_fp8(q8, k8, vt8, qd, kd, vd, causal=True, scale=p.scale)
    torch.cuda.synchronize(dev)
    s = signs.cpu().numpy()
    cq, dq = fp8_quantize(bf16_bits_to_f32(p.q), s)
    ck, dk = fp8_quantize(bf16_bits_to_f32(p.k), s)
    cv, dv = fp8_quantize(bf16_bits_to_f32(p.v), None)
    qq, kk, vv = fp8_dequantize(cq, dq), fp8_dequantize(ck, dk), fp8_dequantize(cv, dv)
    ref_o, ref_lse = attention_fwd(qq, kk, vv, p.scale, True)
    bound, _ = attention_fwd(qq, kk, np.abs(vv), p.scale, True)
    got = o.float().cpu().numpy().astype(np.float64)
    tol = 2.0 ** -4 * bound + 2.0 ** -8 * np.abs(ref_o) + 2e-3
    assert np.all(np.abs(got - ref_o) <= tol), float(np.max(np.abs(got - ref_o) - tol))
    fin = np.isfinite(ref_lse)
    rel = np.abs(lse.cpu().numpy()[fin] - ref_lse[fin]) / np.maximum(1.0, np.abs(ref_lse[fin]))
    assert rel.max() <= 1e-3


def test_rotation_lowers_the_error_with_outlier_channels(fa, dev):
    p = make_dense(1, 2, 2, 512, 512, 128, seed=3, causal=False)
    q, k, v = (bf16_bits_to_f64(x) for x in (p.q, p.k, p.v))
    for t in (q, k):
        t[..., [5, 77]] *= 8.0  # powers of two keep the values bf16
    qb, kb = f64_to_bf16_bits(q), f64_to_bf16_bits(k)
    scale = p.scale / 8.0
    ref, _ = attention_fwd(bf16_bits_to_f64(qb), bf16_bits_to_f64(kb), v, scale, False)
    rms = {}
    for rotate in (False, True):
        o, _ = fa.fwd_fp8_from_bf16(_to_dev(qb, dev), _to_dev(kb, dev), _to_dev(p.v, dev), causal=False,
                                    scale=scale, rotate=rotate, seed=4)
        torch.cuda.synchronize(dev)
        err = o.float().cpu().numpy().astype(np.float64) - ref
        rms[rotate] = math.sqrt(float(np.mean(err ** 2)))
    assert rms[True] < 0.6 * rms[False], rms
    assert rms[True] < 6e-3, rms


def test_non_finite_inputs_follow_the_documented_rule(fa, dev):
    """fa.h states what a NaN or an infinity does to the codes (unrotated):
    a NaN is left out of its slice's maximum and gets a NaN code; an infinity
    makes the slice's descale +inf, its own code NaN and every other code of
    the slice a zero.  Slices without a non-finite element match the oracle."""
    B, H, N, d = 1, 3, 128, 128
    bits = normal_bf16(stream_key(411, 1), (B, H, N, d))
    nan_at, inf_at = (0, 0, 5, 17), (0, 1, 70, 3)
    bits[nan_at] = 0x7FC0   # bf16 quiet NaN
    bits[inf_at] = 0xFF80   # bf16 -inf
    x8, desc = fa.fp8_quantize(_to_dev(bits, dev), None)
    torch.cuda.synchronize(dev)
    got8, got_d = x8.cpu().numpy(), desc.cpu().numpy()
    is_nan_code = lambda c: (c & 0x7F) == 0x7F
    # Slice 0: the NaN element's code is NaN; the rest are the codes of the
    # same slice with that element set to 0 (it is left out of the maximum).
    assert is_nan_code(got8[nan_at])
    clean = bits.copy()
    clean[nan_at] = 0
    clean[inf_at] = 0       # slice 1 is checked against the rule below, not the oracle
    ref8, ref_d = fp8_quantize(bf16_bits_to_f32(clean), None)
    mask = np.ones(got8[0, 0].shape, dtype=bool)
    mask[nan_at[2:]] = False
    assert np.array_equal(got8[0, 0][mask], ref8[0, 0][mask])
    assert got_d[0, 0] == ref_d[0, 0]
    # Slice 1: descale +inf, the infinity's code NaN, every other code a zero.
    assert np.isposinf(got_d[0, 1])
    assert is_nan_code(got8[inf_at])
    rest = np.ones(got8[0, 1].shape, dtype=bool)
    rest[inf_at[2:]] = False
    assert np.all((got8[0, 1][rest] & 0x7F) == 0)
    # Slice 2 is untouched by the others.
    assert np.array_equal(got8[0, 2], ref8[0, 2]) and got_d[0, 2] == ref_d[0, 2]
