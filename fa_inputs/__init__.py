"""Seeded synthetic inputs for the attention forward pass.

This module is shared by the tests, the bench and the smoke check.  It holds
no attention arithmetic: it only draws numbers, rounds them to bf16 and lays
them out.  Both the CUDA path and the oracle consume exactly the bf16 bits it
produces.

Random numbers come from SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) used as a counter-based
generator: draw ``i`` of stream ``key`` is ``mix64(key + (i + 1) * GAMMA)``.
Normal variates use the Box-Muller transform on pairs of 53-bit uniforms.
Values are rounded to float32 and then to bf16 with round-to-nearest-even.

Workload recipes follow the exact-attention interview canvas
("FlashAttention面试讲解", element ``std-text``: Q, K, V of N rows by d) and the
five shapes the library is measured on (see ``WORKLOADS``).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 24


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tensor_id: int) -> int:
    """64-bit key of one named stream (one tensor of one workload)."""
    z = np.array([(seed * 0x100000001B3 + tensor_id * 0x9E37 + 0x51ED27) & ((1 << 64) - 1)],
                 dtype=np.uint64)
    with np.errstate(over="ignore"):
        return int(_mix64(z)[0])


def raw_u64(key: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of stream ``key`` as uint64."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(np.uint64(key) + idx * _GAMMA)


def uniform01(key: int, start: int, count: int) -> np.ndarray:
    """Uniform doubles in [0, 1) with 53 random bits."""
    return (raw_u64(key, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal_f32(key: int, n: int) -> np.ndarray:
    """``n`` standard normal values (Box-Muller), rounded to float32."""
    out = np.empty(n, dtype=np.float32)
    npairs = (n + 1) // 2
    for p0 in range(0, npairs, _CHUNK):
        cnt = min(_CHUNK, npairs - p0)
        u = raw_u64(key, 2 * p0, 2 * cnt)
        u1 = ((u[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
        u2 = (u[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)          # [0, 1)
        r = np.sqrt(-2.0 * np.log(u1))
        t = (2.0 * math.pi) * u2
        z = np.empty(2 * cnt, dtype=np.float64)
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        lo = 2 * p0
        hi = min(n, lo + 2 * cnt)
        out[lo:hi] = z[: hi - lo].astype(np.float32)
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest, ties to even); finite inputs."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    return bf16_bits_to_f32(bits).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> float32 -> bf16 bits (for hand-made test tensors)."""
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float64).astype(np.float32))


def normal_bf16(key: int, shape) -> np.ndarray:
    n = int(np.prod(shape)) if len(shape) else 1
    return f32_to_bf16_bits(normal_f32(key, n)).reshape(shape)


def scale_outliers_bf16(bits: np.ndarray, key: int, frac: float, factor: int) -> np.ndarray:
    """Multiply a seeded ``frac`` of the entries by ``factor`` (a power of two).

    An entry is chosen when its uniform draw from stream ``key`` is below
    ``frac``.  Multiplying a bf16 value by a power of two only moves its
    exponent, so the result is exact and stays bf16.
    """
    assert factor > 0 and (factor & (factor - 1)) == 0
    flat = bits.reshape(-1)
    out = np.empty_like(flat)
    for s0 in range(0, flat.size, _CHUNK):
        s1 = min(flat.size, s0 + _CHUNK)
        sel = uniform01(key, s0, s1 - s0) < frac
        v = bf16_bits_to_f32(flat[s0:s1])
        v = np.where(sel, v * np.float32(factor), v)
        out[s0:s1] = f32_to_bf16_bits(v)
    return out.reshape(bits.shape)


def uniform_ints(key: int, count: int, lo: int, hi: int) -> np.ndarray:
    """``count`` integers uniform on [lo, hi] (inclusive)."""
    u = uniform01(key, 0, count)
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int64)


# --------------------------------------------------------------------------
# FP8 (e4m3) encoding, for the 8-bit forward path's inputs
# --------------------------------------------------------------------------
# OCP 8-bit floating point, E4M3 variant: 1 sign, 4 exponent (bias 7) and 3
# mantissa bits; no infinities; S.1111.111 is NaN, so the largest finite
# magnitude is 1.75 * 2^8 = 448; subnormals go down to 2^-9.

E4M3_MAX = 448.0


def e4m3_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of each e4m3 code (NaN for the two NaN codes)."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = np.where((e == 0xF) & (m == 7), np.nan, val)
    return sign * val


_E4M3_TABLE = e4m3_bits_to_f64(np.arange(128, dtype=np.uint8))  # non-negative codes, increasing


def f64_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round to the nearest e4m3 value (ties to the even code), saturating at
    +-448; finite inputs."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    finite = _E4M3_TABLE[:127]  # codes 0..126 (127 is NaN)
    hi = np.clip(np.searchsorted(finite, a, side="left"), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    dlo = a - finite[lo]
    dhi = finite[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0) & (hi != lo))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(x < 0, code | 0x80, code).astype(np.uint8)


@dataclasses.dataclass
class Fp8Problem:
    """A problem quantized to e4m3 with one scale per (batch, head) slice.

    Dense: q8 [B, Hq, Nq, d], k8 [B, Hkv, Nk, d] and vt8 [B, Hkv, d, Nk] (V
    transposed) are e4m3 codes, and the real inputs are q8 * q_scale[b, h] and
    so on, with scales [B, H].  Packed: q8 [Hq, T, d], k8 [Hkv, T, d],
    vt8 [Hkv, d, T] and scales [H]: the packed tensor counts as one batch.
    Each scale is the slice's max |x| / 448 (1 for an all-zero slice), so the
    slice uses the whole e4m3 range.
    """
    base: "Problem"
    q8: np.ndarray
    k8: np.ndarray
    vt8: np.ndarray
    q_scale: np.ndarray  # [B, Hq] float32 ([Hq] when packed)
    k_scale: np.ndarray  # [B, Hkv] float32
    v_scale: np.ndarray  # [B, Hkv] float32

    def dequantized(self):
        """(q, k, v) as float64 arrays in the problem's layout."""
        if self.q8.ndim == 3:
            q = e4m3_bits_to_f64(self.q8) * self.q_scale.astype(np.float64)[:, None, None]
            k = e4m3_bits_to_f64(self.k8) * self.k_scale.astype(np.float64)[:, None, None]
            vt = e4m3_bits_to_f64(self.vt8) * self.v_scale.astype(np.float64)[:, None, None]
            return q, k, np.swapaxes(vt, 1, 2)
        q = e4m3_bits_to_f64(self.q8) * self.q_scale.astype(np.float64)[:, :, None, None]
        k = e4m3_bits_to_f64(self.k8) * self.k_scale.astype(np.float64)[:, :, None, None]
        vt = e4m3_bits_to_f64(self.vt8) * self.v_scale.astype(np.float64)[:, :, None, None]
        return q, k, np.swapaxes(vt, 2, 3)


def _quantize_slices(x: np.ndarray):
    """Per-[b, h] scale (float32) and e4m3 codes of x / scale."""
    amax = np.max(np.abs(x), axis=(2, 3)) if x.size else np.zeros(x.shape[:2])
    scale = np.where(amax > 0, amax / E4M3_MAX, 1.0).astype(np.float32)
    codes = f64_to_e4m3_bits(x / scale.astype(np.float64)[:, :, None, None])
    return codes, scale


def make_fp8(prob: "Problem") -> Fp8Problem:
    """Quantizes a bf16 problem's Q, K, V to e4m3 (V also transposed); a
    packed problem is quantized as one batch (one scale per head)."""
    q, k, v = (bf16_bits_to_f64(x) for x in (prob.q, prob.k, prob.v))
    packed = prob.cu_seqlens is not None
    if packed:
        q, k, v = q[None], k[None], v[None]
    q8, qs = _quantize_slices(q)
    k8, ks = _quantize_slices(k)
    v8, vs = _quantize_slices(v)
    vt8 = np.ascontiguousarray(np.swapaxes(v8, 2, 3))
    if packed:
        return Fp8Problem(prob, q8[0], k8[0], vt8[0], qs[0], ks[0], vs[0])
    return Fp8Problem(prob, q8, k8, vt8, qs, ks, vs)


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Problem:
    """One attention forward problem as bf16 bit arrays (uint16).

    Dense layout: q [B, Hq, Nq, d], k/v [B, Hkv, Nk, d].
    Packed variable-length layout: q [Hq, T, d], k/v [Hkv, T, d] with
    ``cu_seqlens`` (int32, B+1 entries) giving each sequence's token range;
    then B = number of sequences and Nq = Nk = the longest sequence.
    """
    name: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    scale: float
    cu_seqlens: Optional[np.ndarray] = None

    @property
    def varlen(self) -> bool:
        return self.cu_seqlens is not None

    def seqlens(self):
        if self.cu_seqlens is None:
            return [self.Nq] * self.B
        return [int(self.cu_seqlens[i + 1] - self.cu_seqlens[i]) for i in range(self.B)]

    def flops(self) -> float:
        """4*Hq*Nq*Nk*d per sequence, halved when causal."""
        f = 0.0
        if self.cu_seqlens is None:
            f = 4.0 * self.B * self.Hq * self.Nq * self.Nk * self.d
        else:
            for L in self.seqlens():
                f += 4.0 * self.Hq * L * L * self.d
        return f * (0.5 if self.causal else 1.0)

    def io_bytes(self) -> int:
        """Q, K, V read once and O, LSE written once."""
        return 2 * (self.q.size + self.k.size + self.v.size + self.q.size) + 4 * (self.q.size // self.d)


def make_dense(B, Hq, Hkv, Nq, Nk, d, seed, causal, scale=None, k_outlier_frac=0.0,
               k_outlier_factor=8, name="dense") -> Problem:
    q = normal_bf16(stream_key(seed, 1), (B, Hq, Nq, d))
    k = normal_bf16(stream_key(seed, 2), (B, Hkv, Nk, d))
    v = normal_bf16(stream_key(seed, 3), (B, Hkv, Nk, d))
    if k_outlier_frac > 0:
        k = scale_outliers_bf16(k, stream_key(seed, 4), k_outlier_frac, k_outlier_factor)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return Problem(name, q, k, v, B, Hq, Hkv, Nq, Nk, d, bool(causal), float(scale))


def make_varlen(seqlens, Hq, Hkv, d, seed, causal, scale=None, name="varlen") -> Problem:
    seqlens = [int(x) for x in seqlens]
    cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(seqlens)
    T = int(cu[-1])
    q = normal_bf16(stream_key(seed, 1), (Hq, T, d))
    k = normal_bf16(stream_key(seed, 2), (Hkv, T, d))
    v = normal_bf16(stream_key(seed, 3), (Hkv, T, d))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    L = max(seqlens) if seqlens else 0
    return Problem(name, q, k, v, len(seqlens), Hq, Hkv, L, L, d, bool(causal), float(scale), cu)


def make_dout(prob: Problem, seed: int) -> np.ndarray:
    """Upstream gradient dO for the backward pass: bf16 N(0, 1), O's shape."""
    return normal_bf16(stream_key(seed, 6), prob.q.shape)


def varlen_lengths(seed: int, count: int = 16, lo: int = 256, hi: int = 8192):
    return [int(x) for x in uniform_ints(stream_key(seed, 5), count, lo, hi)]


# The five measured workloads.  "causal" masks are bottom-right aligned.
WORKLOADS = {
    "tiny_b1_h2_n128_d64": dict(kind="dense", B=1, Hq=2, Hkv=2, Nq=128, Nk=128, d=64, seed=1, causal=False),
    "b4_h16_n1024_d64": dict(kind="dense", B=4, Hq=16, Hkv=16, Nq=1024, Nk=1024, d=64, seed=2, causal=False),
    "b4_h16_n1024_d64_causal": dict(kind="dense", B=4, Hq=16, Hkv=16, Nq=1024, Nk=1024, d=64, seed=2, causal=True),
    "b2_h32_n4096_d128_causal": dict(kind="dense", B=2, Hq=32, Hkv=32, Nq=4096, Nk=4096, d=128, seed=3, causal=True),
    "gqa_b1_hq32_hkv8_n16384_d128_causal": dict(kind="dense", B=1, Hq=32, Hkv=8, Nq=16384, Nk=16384, d=128,
                                                seed=4, causal=True, k_outlier_frac=0.01),
    "varlen16_h16_d128_causal": dict(kind="varlen", H=16, d=128, seed=5, causal=True),
    # Decode (split-KV path): a few new tokens per sequence against a long context.
    "decode_b8_hq32_hkv8_nq1_nk32768_d128": dict(kind="dense", B=8, Hq=32, Hkv=8, Nq=1, Nk=32768, d=128, seed=6,
                                                 causal=False),
    "decode_b16_hq32_hkv8_nq4_nk8192_d128_causal": dict(kind="dense", B=16, Hq=32, Hkv=8, Nq=4, Nk=8192, d=128,
                                                        seed=7, causal=True),
}

HEADLINE = "b2_h32_n4096_d128_causal"
# Workloads the 8-bit forward path is measured on (quantized with make_fp8).
FP8_WORKLOADS = ("b2_h32_n4096_d128_causal", "gqa_b1_hq32_hkv8_n16384_d128_causal")


def make_workload(name: str) -> Problem:
    w = dict(WORKLOADS[name])
    kind = w.pop("kind")
    if kind == "dense":
        return make_dense(name=name, **w)
    lens = varlen_lengths(w["seed"])
    return make_varlen(lens, w["H"], w["H"], w["d"], w["seed"], w["causal"], name=name)
