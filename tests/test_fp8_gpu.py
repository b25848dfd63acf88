"""GPU parity of the 8-bit forward (fa_fwd_fp8) against the fp64 oracle.

The oracle runs the plain definition on the dequantized inputs (e4m3 code x
descale, exactly representable in float64), so the only departure of the
kernel from it is P rounded to e4m3 before the P V product, plus fp32
accumulation and the bf16 output.  Rounding changes each term p_j v_j by at
most 2^-4 of itself, so for every output element

    |O_gpu - O_ref| <= 2^-4 * (sum_j p_j |v_j|) / l + 2^-8 |O_ref| + 2e-3,

where the first term is the oracle's attention with |V| in place of V, the
second the bf16 rounding of O and the last covers fp32 accumulation and the
exponential.  LSE is formed from the unrounded p and keeps the fp16-path
tolerance (1e-3 relative).
"""
import numpy as np
import pytest
import torch

from fa_inputs import make_dense, make_fp8, make_varlen, make_workload
from fa_testutil import LSE_RTOL
from oracle import attention_fwd

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


def _run(fa, f8, dev):
    u8 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
    p = f8.base
    o, lse = fa.fwd_fp8(u8(f8.q8), u8(f8.k8), u8(f8.vt8), f32(f8.q_scale), f32(f8.k_scale), f32(f8.v_scale),
                        causal=p.causal, scale=p.scale)
    torch.cuda.synchronize(dev)
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _check(o, lse, ref_o, ref_lse, bound_o, what):
    assert np.all(np.isfinite(o)), what
    inf = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), inf), what + ": -inf LSE pattern"
    assert np.all(o[inf] == 0.0), what
    tol = 2.0 ** -4 * bound_o + 2.0 ** -8 * np.abs(ref_o) + 2e-3
    err = np.abs(o - ref_o)
    bad = err > tol
    assert not bad.any(), "%s: %d elements over the bound, worst excess %.4g" % (what, bad.sum(), (err - tol).max())
    fin = ~inf
    if fin.any():
        rel = np.abs(lse[fin] - ref_lse[fin]) / np.maximum(1.0, np.abs(ref_lse[fin]))
        assert rel.max() <= LSE_RTOL, "%s: LSE %.3g" % (what, rel.max())


FP8 = [
    # (B, Hq, Hkv, Nq, Nk, causal); d = 128, Nk a multiple of 16
    (1, 2, 2, 128, 128, False),
    (1, 4, 2, 200, 256, False),     # GQA, ragged query tile
    (2, 4, 2, 300, 304, True),      # causal, ragged tiles
    (1, 2, 2, 130, 400, True),      # Nq < Nk, bottom-right
    (1, 2, 2, 400, 208, True),      # Nq > Nk: early rows see no key
    (1, 2, 1, 64, 16, False),       # one short K/V tile
    (1, 8, 1, 640, 640, True),      # MQA, several units
    (3, 20, 5, 700, 1008, True),    # more units than SMs, GQA, Nq < Nk
]


@pytest.mark.parametrize("shape", FP8, ids=["-".join(map(str, s)) for s in FP8])
def test_fp8_matches_oracle(fa, dev, shape):
    B, Hq, Hkv, Nq, Nk, causal = shape
    p = make_dense(B, Hq, Hkv, Nq, Nk, 128, seed=sum(shape) + 500, causal=causal, name="fp8")
    f8 = make_fp8(p)
    o, lse = _run(fa, f8, dev)
    q, k, v = f8.dequantized()
    ref_o, ref_lse = attention_fwd(q, k, v, p.scale, causal)
    bound, _ = attention_fwd(q, k, np.abs(v), p.scale, causal)
    _check(o, lse, ref_o, ref_lse, bound, "fp8 %s" % (shape,))


def test_fp8_is_deterministic(fa, dev):
    p = make_dense(1, 4, 2, 384, 384, 128, seed=91, causal=True)
    f8 = make_fp8(p)
    a = _run(fa, f8, dev)
    b = _run(fa, f8, dev)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_fp8_headline_full_size(fa, dev):
    """The B2 H32 N4096 d128 causal workload, quantized: every element of O
    and LSE against the oracle, one (batch, head) at a time."""
    p = make_workload("b2_h32_n4096_d128_causal")
    f8 = make_fp8(p)
    o, lse = _run(fa, f8, dev)
    q, k, v = f8.dequantized()
    g = p.Hq // p.Hkv
    for b in range(p.B):
        for h in range(p.Hq):
            kq, kk = (b, h), (b, h // g)
            qs, ks, vs = q[kq[0]:kq[0] + 1, kq[1]:kq[1] + 1], k[kk[0]:kk[0] + 1, kk[1]:kk[1] + 1], \
                v[kk[0]:kk[0] + 1, kk[1]:kk[1] + 1]
            ref_o, ref_lse = attention_fwd(qs, ks, vs, p.scale, True)
            bound, _ = attention_fwd(qs, ks, np.abs(vs), p.scale, True)
            _check(o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], ref_o, ref_lse, bound,
                   "fp8 headline b=%d h=%d" % (b, h))


FP8_D64 = [
    # (B, Hq, Hkv, Nq, Nk, causal); d = 64 (rows of 64 bytes: the 64-byte swizzle)
    (1, 2, 2, 128, 128, False),
    (1, 4, 2, 200, 256, False),
    (2, 4, 2, 300, 304, True),
    (1, 2, 2, 400, 208, True),
    (1, 8, 1, 640, 640, True),
    (2, 40, 8, 700, 704, False),    # more units than SMs
]


@pytest.mark.parametrize("shape", FP8_D64, ids=["d64-" + "-".join(map(str, s)) for s in FP8_D64])
def test_fp8_d64_matches_oracle(fa, dev, shape):
    B, Hq, Hkv, Nq, Nk, causal = shape
    p = make_dense(B, Hq, Hkv, Nq, Nk, 64, seed=sum(shape) + 700, causal=causal, name="fp8 d64")
    f8 = make_fp8(p)
    o, lse = _run(fa, f8, dev)
    q, k, v = f8.dequantized()
    ref_o, ref_lse = attention_fwd(q, k, v, p.scale, causal)
    bound, _ = attention_fwd(q, k, np.abs(v), p.scale, causal)
    _check(o, lse, ref_o, ref_lse, bound, "fp8 d64 %s" % (shape,))


def _run_packed(fa, f8, dev):
    u8 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
    p = f8.base
    cu = torch.from_numpy(p.cu_seqlens).to(dev)
    o, lse = fa.fwd_fp8(u8(f8.q8), u8(f8.k8), u8(f8.vt8), f32(f8.q_scale), f32(f8.k_scale), f32(f8.v_scale),
                        causal=p.causal, scale=p.scale, cu_seqlens=cu)
    torch.cuda.synchronize(dev)
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


# Sequence starts that are not multiples of 16 tokens: the kernel reads each
# sequence's key tiles from the multiple of 16 below its start and masks the
# keys before it.  Every total is a multiple of 16 (rows of V^T are T bytes).
FP8_PACKED = [
    ([1, 127, 128, 129, 0, 300, 256, 700, 7], 4, 2, 128, True),
    ([1, 127, 128, 129, 0, 300, 256, 700, 7], 4, 2, 128, False),
    ([17, 5, 513, 3, 1000, 14], 2, 2, 64, True),
    ([0, 0, 64], 1, 1, 64, False),
]


@pytest.mark.parametrize("case", FP8_PACKED, ids=["p%d" % i for i in range(len(FP8_PACKED))])
def test_fp8_packed_matches_oracle(fa, dev, case):
    lens, Hq, Hkv, d, causal = case
    assert sum(lens) % 16 == 0
    p = make_varlen(lens, Hq, Hkv, d, seed=len(lens) + d + 900, causal=causal)
    f8 = make_fp8(p)
    o, lse = _run_packed(fa, f8, dev)
    q, k, v = f8.dequantized()
    ref_o, ref_lse = attention_fwd(q, k, v, p.scale, causal, cu_seqlens=p.cu_seqlens)
    bound, _ = attention_fwd(q, k, np.abs(v), p.scale, causal, cu_seqlens=p.cu_seqlens)
    _check(o, lse, ref_o, ref_lse, bound, "fp8 packed %s" % (lens,))


def test_fp8_d64_growing_scores_force_rescales(fa, dev):
    """Scores that grow along the key axis move the running max by more than
    the 8-bit rescale threshold in every K/V tile.  At d = 64 the next QK
    product runs ahead of the previous P V, so each correction of O first
    waits for that product."""
    from fa_inputs import f64_to_bf16_bits
    N, d = 1024, 64
    q = np.full((1, 2, N, d), 0.25)
    ramp = np.linspace(0.0, 40.0, N)[None, None, :, None]
    k = np.broadcast_to(ramp, (1, 2, N, d)) + 0.01 * np.random.default_rng(0).standard_normal((1, 2, N, d))
    v = np.random.default_rng(1).standard_normal((1, 2, N, d))
    for causal in (False, True):
        p = make_dense(1, 2, 2, N, N, d, seed=0, causal=causal)
        p.q, p.k, p.v = (f64_to_bf16_bits(x) for x in (q, k, v))
        p.scale = 1.0 / np.sqrt(d)
        f8 = make_fp8(p)
        o, lse = _run(fa, f8, dev)
        qq, kk, vv = f8.dequantized()
        ref_o, ref_lse = attention_fwd(qq, kk, vv, p.scale, causal)
        bound, _ = attention_fwd(qq, kk, np.abs(vv), p.scale, causal)
        _check(o, lse, ref_o, ref_lse, bound, "fp8 d64 growing scores causal=%s" % causal)


def test_fp8_d64_from_bf16_with_rotation(fa, dev):
    """The quantizer and the 8-bit forward at d = 64 together: within the
    8-bit bound of the oracle on the same dequantized, rotated inputs."""
    from oracle.fp8 import fp8_dequantize, fp8_quantize
    from fa_inputs import bf16_bits_to_f32
    p = make_dense(1, 4, 2, 300, 256, 64, seed=41, causal=True)
    tb = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)
    signs = fa.hadamard_signs(64, 5, dev)
    q8, qd = fa.fp8_quantize(tb(p.q), signs)
    k8, kd = fa.fp8_quantize(tb(p.k), signs)
    vt8, vd = fa.fp8_quantize(tb(p.v), None, transpose=True)
    o, lse = fa.fwd_fp8(q8, k8, vt8, qd, kd, vd, causal=True, scale=p.scale)
    torch.cuda.synchronize(dev)
    s = signs.cpu().numpy()
    cq, dq = fp8_quantize(bf16_bits_to_f32(p.q), s)
    ck, dk = fp8_quantize(bf16_bits_to_f32(p.k), s)
    cv, dv = fp8_quantize(bf16_bits_to_f32(p.v), None)
    qq, kk, vv = fp8_dequantize(cq, dq), fp8_dequantize(ck, dk), fp8_dequantize(cv, dv)
    ref_o, ref_lse = attention_fwd(qq, kk, vv, p.scale, True)
    bound, _ = attention_fwd(qq, kk, np.abs(vv), p.scale, True)
    _check(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ref_o, ref_lse, bound,
           "fp8 d64 quantized")
