"""GPU parity of the forward kernels with software exponentials switched on.

fa_debug_soft_exp(1) selects the kernel instantiation that computes one
exponential pair in every two of each K/V tile without a mask with the
FMA-pipe 2^x (range reduction plus a degree-3 minimax polynomial, relative
error below 7.5e-5; the "software exp" of the interview canvas's Blackwell
notes, element v4-card-body) instead of the exp unit.  That error is far
below the bf16 rounding of P (2^-9), so the results must meet the same
tolerances as the default path, against the same oracle.
"""
import numpy as np
import pytest
import torch

from fa_inputs import make_dense, make_fp8, make_varlen, make_workload
from fa_testutil import compare, compare_per_head, oracle_full, run_gpu, to_dev
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
def _soft_on(fa):
    fa.fa_device_status()
    fa.fa_debug_soft_exp(1)
    try:
        yield
    finally:
        fa.fa_debug_soft_exp(0)
    assert fa.fa_device_status() == 0, "a kernel wait timed out"


SHAPES = [
    # (B, Hq, Hkv, Nq, Nk, d, causal)
    (2, 3, 3, 200, 200, 128, True),
    (1, 4, 2, 640, 640, 128, False),
    (2, 8, 2, 257, 257, 64, True),
    (3, 5, 5, 384, 640, 64, False),
    (1, 2, 2, 300, 77, 128, True),
]


@pytest.mark.parametrize("shape", SHAPES, ids=["-".join(map(str, s)) for s in SHAPES])
def test_soft_exp_matches_oracle(fa, dev, shape):
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    prob = make_dense(B, Hq, Hkv, Nq, Nk, d, seed=sum(shape) + 7, causal=causal, name="soft")
    o, lse = run_gpu(fa, prob, dev)
    ref_o, ref_lse = oracle_full(prob)
    compare(o, lse, ref_o, ref_lse, "soft exp %s" % (shape,))


def test_soft_exp_varlen(fa, dev):
    prob = make_varlen([1, 127, 128, 129, 0, 300, 256, 700], 4, 2, 128, seed=31, causal=True)
    o, lse = run_gpu(fa, prob, dev)
    ref_o, ref_lse = oracle_full(prob)
    compare(o, lse, ref_o, ref_lse, "soft exp varlen")


def test_soft_exp_path_is_taken(fa, dev):
    """The hook selects a different kernel: its rounding of P differs from the
    exp unit's somewhere, while both stay within tolerance."""
    prob = make_dense(1, 4, 4, 1024, 1024, 128, seed=33, causal=False)
    q, k, v = (to_dev(x, dev) for x in (prob.q, prob.k, prob.v))
    o_soft, l_soft = fa.fwd(q, k, v)
    fa.fa_debug_soft_exp(0)
    o_mufu, l_mufu = fa.fwd(q, k, v)
    fa.fa_debug_soft_exp(1)
    torch.cuda.synchronize(dev)
    assert not torch.equal(o_soft, o_mufu)
    ref_o, ref_lse = oracle_full(prob)
    for o, l in ((o_soft, l_soft), (o_mufu, l_mufu)):
        compare(o.float().cpu().numpy().astype(np.float64), l.cpu().numpy().astype(np.float64), ref_o, ref_lse,
                "soft/mufu")


def test_soft_exp_headline_full_size(fa, dev):
    prob = make_workload("b2_h32_n4096_d128_causal")
    o, lse = run_gpu(fa, prob, dev, keep_on_device=True)
    compare_per_head(o, lse, prob, "soft exp headline")


def test_soft_exp_fp8(fa, dev):
    """The 8-bit forward's software-exponential instantiation, under the
    8-bit path's per-element bound (see test_fp8_gpu)."""
    p = make_dense(2, 4, 2, 300, 304, 128, seed=77, causal=True, name="fp8 soft")
    f8 = make_fp8(p)
    u8 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
    o, lse = fa.fwd_fp8(u8(f8.q8), u8(f8.k8), u8(f8.vt8), f32(f8.q_scale), f32(f8.k_scale), f32(f8.v_scale),
                        causal=True, scale=p.scale)
    torch.cuda.synchronize(dev)
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    q, k, v = f8.dequantized()
    ref_o, ref_lse = attention_fwd(q, k, v, p.scale, True)
    bound, _ = attention_fwd(q, k, np.abs(v), p.scale, True)
    tol = 2.0 ** -4 * bound + 2.0 ** -8 * np.abs(ref_o) + 2e-3
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    assert not (np.abs(o - ref_o) > tol).any()
    fin = np.isfinite(ref_lse)
    assert (np.abs(lse[fin] - ref_lse[fin]) / np.maximum(1.0, np.abs(ref_lse[fin]))).max() <= 1e-3
