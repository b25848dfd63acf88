"""GPU parity of the CTA-pair forward kernel (tcgen05 cta_group::2), which
fa_debug_fwd_pair(1) selects for bf16 problems with d = 128.

Two CTAs of a cluster share every tensor-core product (M = 256): each holds
its own 128 query rows of a product tile and half of each K tile (64 keys)
and V tile (64 head dims), the even CTA issues the products for both, and
the two CTAs hand S, P and O over through each other's barriers.  The
interview canvas's Blackwell notes (element v4-card-body) name these 2-CTA
products.  The kernel must give the same results as the single-CTA one
within the same tolerances, against the same oracle: every element, at
ragged and full sizes.
"""
import numpy as np
import pytest
import torch

from fa_inputs import make_dense, make_varlen, make_workload
from fa_testutil import compare, compare_per_head, oracle_full, run_gpu, to_dev

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
def _pair_on(fa):
    fa.fa_device_status()
    fa.fa_debug_fwd_pair(1)
    try:
        yield
    finally:
        fa.fa_debug_fwd_pair(0)
    assert fa.fa_device_status() == 0, "a kernel wait timed out"


SHAPES = [
    # (B, Hq, Hkv, Nq, Nk, d, causal)
    (1, 1, 1, 512, 512, 128, False),     # one pair unit
    (2, 3, 3, 200, 200, 128, True),      # the odd CTA's rows all past the end in one product tile
    (1, 4, 2, 700, 300, 128, True),      # Nq > Nk: rows with no visible key
    (1, 2, 1, 77, 300, 128, True),       # Nq < Nk, shorter than one CTA's tile
    (1, 32, 1, 130, 130, 128, True),     # MQA
    (2, 8, 2, 1025, 1025, 128, False),   # pair unit + 1 row
    (1, 2, 2, 1, 1, 128, False),         # g * Nq = 1: fa_fwd hands this to the split-KV path (the hook does not apply)
    (1, 4, 4, 300, 0, 128, True),        # no keys
]


@pytest.mark.parametrize("shape", SHAPES, ids=["-".join(map(str, s)) for s in SHAPES])
def test_pair_matches_oracle(fa, dev, shape):
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    prob = make_dense(B, Hq, Hkv, Nq, Nk, d, seed=sum(shape) + 3, causal=causal, name="pair")
    o, lse = run_gpu(fa, prob, dev)
    if Nk == 0:
        assert np.all(o == 0.0) and np.all(np.isneginf(lse))
        return
    ref_o, ref_lse = oracle_full(prob)
    compare(o, lse, ref_o, ref_lse, "pair %s" % (shape,))


def test_pair_varlen(fa, dev):
    prob = make_varlen([1, 127, 128, 129, 0, 300, 256, 700, 513], 4, 2, 128, seed=7, causal=True)
    o, lse = run_gpu(fa, prob, dev)
    ref_o, ref_lse = oracle_full(prob)
    compare(o, lse, ref_o, ref_lse, "pair varlen")


def test_pair_output_canaries(fa, dev):
    """Writes stay inside O and LSE on the pair path too."""
    lens = [1, 130, 0, 255, 257, 600]
    prob = make_varlen(lens, 3, 1, 128, seed=9, causal=True)
    q, k, v = (to_dev(x, dev) for x in (prob.q, prob.k, prob.v))
    cu = torch.from_numpy(prob.cu_seqlens).to(dev)
    T, G = int(prob.cu_seqlens[-1]), 4096
    obuf = torch.full((G + 3 * T * 128 + G,), 7.0, dtype=torch.bfloat16, device=dev)
    lbuf = torch.full((G + 3 * T + G,), 7.0, dtype=torch.float32, device=dev)
    o = obuf[G:G + 3 * T * 128].view(3, T, 128)
    l = lbuf[G:G + 3 * T].view(3, T)
    fa.fwd(q, k, v, causal=True, cu_seqlens=cu, out=o, lse=l)
    torch.cuda.synchronize(dev)
    assert torch.all(obuf[:G] == 7.0) and torch.all(obuf[G + 3 * T * 128:] == 7.0)
    assert torch.all(lbuf[:G] == 7.0) and torch.all(lbuf[G + 3 * T:] == 7.0)
    ref_o, ref_lse = oracle_full(prob)
    compare(o.float().cpu().numpy().astype(np.float64), l.cpu().numpy().astype(np.float64), ref_o, ref_lse,
            "pair canary")


def test_pair_headline_full_size(fa, dev):
    prob = make_workload("b2_h32_n4096_d128_causal")
    o, lse = run_gpu(fa, prob, dev, keep_on_device=True)
    compare_per_head(o, lse, prob, "pair headline")


def test_pair_withheld_copy_times_out(fa, dev):
    """The bounded waits of both CTAs of a pair run out cleanly, and the
    context stays usable."""
    prob = make_dense(1, 4, 4, 1024, 1024, 128, seed=17, causal=True)
    fa.fa_device_status()
    fa.fa_debug_fault_injection(1, 0.05)
    try:
        run_gpu(fa, prob, dev)
    finally:
        fa.fa_debug_fault_injection(0, 0.0)
    bits = fa.fa_device_status()
    assert bits & 0b11 and bits & ~0x1f == 0, "bits=%#x" % bits
    o, lse = run_gpu(fa, prob, dev)
    ref_o, ref_lse = oracle_full(prob)
    compare(o, lse, ref_o, ref_lse, "pair after fault injection")
