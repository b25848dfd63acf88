"""GPU parity of the backward pass (fa_bwd) against the fp64 oracle.

Tolerance (derived from the arithmetic, the target states none for the
gradients): P and dS are rounded to bf16 (unit roundoff u = 2^-9) before the
fp32-accumulating tensor-core products, the outputs are rounded to bf16, and
delta is formed from the forward pass's bf16 O.  Each gradient X must satisfy
max |X_gpu - X_ref| <= 2e-2 * max |X_ref| (about 10 u, leaving room for
cancellation in the sums) and ||X_gpu - X_ref||_F <= 1e-2 * ||X_ref||_F.
"""
import numpy as np
import pytest
import torch

from fa_inputs import bf16_bits_to_f64, make_dense, make_dout, make_varlen, make_workload
from fa_testutil import to_dev
from oracle import attention_bwd, attention_bwd_keys, attention_bwd_rows

pytestmark = pytest.mark.gpu

MAX_REL = 2e-2
FRO_REL = 1e-2


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


def _run(fa, prob, do_bits, dev):
    q, k, v, do = (to_dev(x, dev) for x in (prob.q, prob.k, prob.v, do_bits))
    o, lse = fa.fwd(q, k, v, causal=prob.causal, scale=prob.scale)
    dq, dk, dv, delta = fa.bwd(q, k, v, o, lse, do, causal=prob.causal, scale=prob.scale)
    torch.cuda.synchronize(dev)
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    return f(dq), f(dk), f(dv), f(delta)


def _check(name, got, ref):
    assert got.shape == ref.shape, name
    assert np.all(np.isfinite(got)), name + ": non-finite"
    big = float(np.max(np.abs(ref))) if ref.size else 0.0
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    if big == 0.0:
        assert err == 0.0, "%s: expected exact zeros, max |err| %.3g" % (name, err)
        return
    fro = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert err <= MAX_REL * big, "%s: max|err| %.4g > %.1e * %.4g" % (name, err, MAX_REL, big)
    assert fro <= FRO_REL, "%s: relative Frobenius error %.4g" % (name, fro)


BWD = [
    # (B, Hq, Hkv, Nq, Nk, d, causal)
    (1, 2, 2, 128, 128, 64, False),      # one tile
    (1, 2, 1, 200, 300, 128, False),     # GQA, ragged tiles
    (2, 4, 2, 256, 256, 128, True),      # causal, GQA, two tiles
    (1, 2, 2, 300, 200, 64, True),       # Nq > Nk: early rows see no key
    (1, 2, 2, 130, 390, 128, True),      # Nq < Nk, bottom-right causal
    (1, 4, 1, 512, 512, 128, True),      # MQA, several tiles
    (1, 1, 1, 1, 5, 64, False),          # a single query row
    (2, 3, 3, 257, 129, 64, False),      # ragged d = 64
    (2, 16, 16, 1300, 1300, 64, True),   # more units than SMs in both kernels: host-built worker lists
    (1, 24, 6, 1000, 1500, 128, True),   # the same for the dQ kernel, GQA, Nq < Nk
]


@pytest.mark.parametrize("shape", BWD, ids=["-".join(map(str, s)) for s in BWD])
def test_bwd_matches_oracle(fa, dev, shape):
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    prob = make_dense(B, Hq, Hkv, Nq, Nk, d, seed=sum(shape) + 300, causal=causal, name="bwd")
    do_bits = make_dout(prob, sum(shape) + 301)
    dq, dk, dv, delta = _run(fa, prob, do_bits, dev)
    q, k, v, do = (bf16_bits_to_f64(x) for x in (prob.q, prob.k, prob.v, do_bits))
    rq, rk, rv, rd = attention_bwd(q, k, v, do, prob.scale, causal)
    _check("dq", dq, rq)
    _check("dk", dk, rk)
    _check("dv", dv, rv)
    _check("delta", delta, rd)


def test_bwd_is_deterministic(fa, dev):
    prob = make_dense(1, 4, 2, 384, 384, 128, seed=77, causal=True, name="det")
    do_bits = make_dout(prob, 78)
    a = _run(fa, prob, do_bits, dev)
    b = _run(fa, prob, do_bits, dev)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_bwd_without_keys(fa, dev):
    """Nk = 0: every row sees no key, so O = 0, dQ = 0 and delta = 0."""
    prob = make_dense(1, 2, 2, 130, 0, 64, seed=5, causal=False, name="nokeys")
    q = to_dev(prob.q, dev)
    do = to_dev(make_dout(prob, 6), dev)
    k = torch.empty((1, 2, 0, 64), dtype=torch.bfloat16, device=dev)
    o, lse = fa.fwd(q, k, k, scale=prob.scale)
    dq, dk, dv, delta = fa.bwd(q, k, k, o, lse, do, scale=prob.scale)
    torch.cuda.synchronize(dev)
    assert torch.all(dq == 0) and torch.all(delta == 0)
    assert dk.numel() == 0 and dv.numel() == 0


@pytest.mark.parametrize("name", ["b2_h32_n4096_d128_causal"])
def test_bwd_workload_sampled(fa, dev, name):
    """The bench workload at full size, checked on sampled query rows (dQ, delta)
    and sampled keys (dK, dV) that the oracle computes one by one."""
    prob = make_workload(name)
    do_bits = make_dout(prob, 1000)
    dq, dk, dv, delta = _run(fa, prob, do_bits, dev)
    q, k, v, do = (bf16_bits_to_f64(x) for x in (prob.q, prob.k, prob.v, do_bits))
    rng = np.random.default_rng(4)
    rows = sorted({0, 127, 128, prob.Nq - 1, *map(int, rng.integers(prob.Nq, size=4))})
    for b, h in ((0, 0), (1, prob.Hq - 1)):
        rq, rd = attention_bwd_rows(q, k, v, do, prob.scale, prob.causal, b, h, rows)
        _check("dq[%d,%d]" % (b, h), dq[b, h, rows], rq)
        _check("delta[%d,%d]" % (b, h), delta[b, h, rows], rd)
    keys = sorted({0, 127, 128, prob.Nk - 1, *map(int, rng.integers(prob.Nk, size=4))})
    for b, kvh in ((0, 3),):
        rk, rv = attention_bwd_keys(q, k, v, do, prob.scale, prob.causal, b, kvh, keys)
        _check("dk[%d,%d]" % (b, kvh), dk[b, kvh, keys], rk)
        _check("dv[%d,%d]" % (b, kvh), dv[b, kvh, keys], rv)


def test_bwd_workload_full_size(fa, dev):
    """The bench workload (B2 H32 N4096 d128 causal) at full size: every
    element of dQ, dK, dV and delta against the oracle, one (batch, head) at a
    time (one query head per key/value head here, so each slice is a whole
    problem of its own)."""
    prob = make_workload("b2_h32_n4096_d128_causal")
    assert prob.Hq == prob.Hkv
    do_bits = make_dout(prob, 1000)
    dq, dk, dv, delta = _run(fa, prob, do_bits, dev)
    q, k, v, do = (bf16_bits_to_f64(x) for x in (prob.q, prob.k, prob.v, do_bits))
    for b in range(prob.B):
        for h in range(prob.Hq):
            sl = (slice(b, b + 1), slice(h, h + 1))
            rq, rk, rv, rd = attention_bwd(q[sl], k[sl], v[sl], do[sl], prob.scale, prob.causal)
            _check("dq[%d,%d]" % (b, h), dq[sl], rq)
            _check("dk[%d,%d]" % (b, h), dk[sl], rk)
            _check("dv[%d,%d]" % (b, h), dv[sl], rv)
            _check("delta[%d,%d]" % (b, h), delta[sl], rd)


@pytest.mark.parametrize("lens,hq,hkv,d,causal", [
    ([5, 130, 1, 256, 300], 4, 2, 128, True),
    ([0, 129, 128, 64], 2, 2, 64, False),
    ([700, 33], 4, 1, 128, True),
])
def test_bwd_varlen_matches_oracle(fa, dev, lens, hq, hkv, d, causal):
    """Packed sequences (lengths 0, 1, ragged, tile multiples): every sequence's
    gradients involve its own tokens only."""
    prob = make_varlen(lens, hq, hkv, d, seed=sum(lens) + hq, causal=causal, name="bwd_varlen")
    do_bits = make_dout(prob, sum(lens) + 7)
    q, k, v, do = (to_dev(x, dev) for x in (prob.q, prob.k, prob.v, do_bits))
    cu = torch.from_numpy(prob.cu_seqlens).to(dev)
    o, lse = fa.fwd(q, k, v, causal=causal, scale=prob.scale, cu_seqlens=cu)
    dq, dk, dv, delta = fa.bwd(q, k, v, o, lse, do, causal=causal, scale=prob.scale, cu_seqlens=cu)
    torch.cuda.synchronize(dev)
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    qq, kk, vv, dd = (bf16_bits_to_f64(x) for x in (prob.q, prob.k, prob.v, do_bits))
    rq, rk, rv, rd = attention_bwd(qq, kk, vv, dd, prob.scale, causal, cu_seqlens=prob.cu_seqlens)
    _check("dq", f(dq), rq)
    _check("dk", f(dk), rk)
    _check("dv", f(dv), rv)
    _check("delta", f(delta), rd)
