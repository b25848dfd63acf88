"""Failure detection without a GPU fault: a copy that never arrives makes the
kernels' bounded waits run out; each kernel must report it in its device
status bits, exit cleanly and leave the context usable.

Modes of fa_debug_fault_injection (include/fa.h): 1 the forward kernel's K/V
producer, 2 the split-KV kernel's producer, 3 the backward dQ kernel's K/V
producer, 4 the backward dK/dV kernel's Q/dO producer, 5 the one-launch
quantizer withhold their first copy.  Each case then runs the same problem
again and checks it against the oracle."""
import numpy as np
import pytest
import torch

from fa_inputs import bf16_bits_to_f64, make_dense, make_dout
from fa_testutil import run_gpu, oracle_full, compare, to_dev


def test_hook_argument_checks():
    import exact_attention_42_gb300 as fa
    fa.build()
    with pytest.raises(fa.FaError):
        fa.fa_debug_fault_injection(6, 0.1)
    with pytest.raises(fa.FaError):
        fa.fa_debug_fault_injection(-1, 0.1)
    with pytest.raises(fa.FaError):
        fa.fa_debug_fault_injection(1, 11.0)
    with pytest.raises(fa.FaError):
        fa.fa_debug_fault_injection(1, float("nan"))
    fa.fa_debug_fault_injection(0, 0.0)
    with pytest.raises(fa.FaError):
        fa.fa_debug_soft_exp(2)
    fa.fa_debug_soft_exp(0)


def _inject(fa, mode, fn):
    fa.fa_device_status()
    fa.fa_debug_fault_injection(mode, 0.05)
    try:
        fn()          # returns once the kernel has given up and exited
    finally:
        fa.fa_debug_fault_injection(0, 0.0)
    return fa.fa_device_status()


@pytest.mark.gpu
def test_withheld_copy_times_out_and_context_survives():
    import exact_attention_42_gb300 as fa
    fa.build()
    dev = torch.device("cuda", 0)
    prob = make_dense(1, 4, 4, 512, 512, 64, seed=17, causal=True)
    bits = _inject(fa, 1, lambda: run_gpu(fa, prob, dev))
    # Whichever role's bounded wait ran out first raised the abort: the K/V
    # producer (bit 0, its slot is never released) or the MMA issuer (bit 1,
    # the copy never lands).  Roles that then saw the abort flag leave quietly.
    assert bits & 0b11, "a bounded wait should have run out (bits=%#x)" % bits
    assert bits & ~0x1f == 0, "only forward roles may report (bits=%#x)" % bits
    # The same process keeps working.
    o, lse = run_gpu(fa, prob, dev)
    ref_o, ref_lse = oracle_full(prob)
    compare(o, lse, ref_o, ref_lse, "after fault injection")
    assert fa.fa_device_status() == 0


@pytest.mark.gpu
def test_decode_withheld_tile_times_out_and_context_survives():
    import exact_attention_42_gb300 as fa
    fa.build()
    dev = torch.device("cuda", 0)
    prob = make_dense(2, 8, 2, 1, 3000, 128, seed=18, causal=False)   # split-KV path: g * Nq = 4
    # The forward kernel is not affected by mode 2: a dense problem first.
    dense = make_dense(1, 2, 2, 256, 256, 64, seed=19, causal=True)
    assert _inject(fa, 2, lambda: run_gpu(fa, dense, dev)) == 0
    bits = _inject(fa, 2, lambda: run_gpu(fa, prob, dev))
    assert bits == 1 << 8, "the split-KV kernel should report bit 8 (bits=%#x)" % bits
    o, lse = run_gpu(fa, prob, dev)
    ref_o, ref_lse = oracle_full(prob)
    compare(o, lse, ref_o, ref_lse, "decode after fault injection")
    assert fa.fa_device_status() == 0


def _bwd_case(fa, dev, prob, do_bits):
    q, k, v, do = (to_dev(x, dev) for x in (prob.q, prob.k, prob.v, do_bits))
    o, lse = fa.fwd(q, k, v, causal=prob.causal, scale=prob.scale)
    torch.cuda.synchronize(dev)
    assert fa.fa_device_status() == 0

    def run():
        g = fa.bwd(q, k, v, o, lse, do, causal=prob.causal, scale=prob.scale)
        torch.cuda.synchronize(dev)
        return g
    return run


@pytest.mark.gpu
@pytest.mark.parametrize("mode,mask,name", [(3, 0b111 << 9, "dQ"), (4, 0b111 << 13, "dK/dV")])
def test_bwd_withheld_fill_times_out_and_context_survives(mode, mask, name):
    import exact_attention_42_gb300 as fa
    from oracle import attention_bwd
    fa.build()
    dev = torch.device("cuda", 0)
    prob = make_dense(1, 4, 2, 384, 384, 128, seed=20 + mode, causal=True)
    do_bits = make_dout(prob, 7)
    run = _bwd_case(fa, dev, prob, do_bits)
    bits = _inject(fa, mode, run)
    assert bits & mask, "the %s kernel should report a time-out (bits=%#x)" % (name, bits)
    assert bits & ~mask == 0, "only the %s kernel may report (bits=%#x)" % (name, bits)
    dq, dk, dv, delta = (t.float().cpu().numpy().astype(np.float64) for t in run())
    assert fa.fa_device_status() == 0
    f = bf16_bits_to_f64
    ref = attention_bwd(f(prob.q), f(prob.k), f(prob.v), f(do_bits), prob.scale, prob.causal)
    for nm, got, want in zip(("dq", "dk", "dv", "delta"), (dq, dk, dv, delta), ref):
        big = float(np.max(np.abs(want)))
        err = float(np.max(np.abs(got - want)))
        assert err <= 2e-2 * big, "%s after fault injection: max err %.3g of max |ref| %.3g" % (nm, err, big)


@pytest.mark.gpu
def test_quantizer_withheld_copy_times_out_and_context_survives():
    import exact_attention_42_gb300 as fa
    from fa_inputs import bf16_bits_to_f32, normal_bf16, stream_key
    from oracle.fp8 import fp8_quantize
    fa.build()
    dev = torch.device("cuda", 0)
    bits = normal_bf16(stream_key(77, 1), (2, 3, 700, 128))   # 700 rows: the one-launch path
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    def run():
        r = fa.fp8_quantize(x, None)
        torch.cuda.synchronize(dev)
        return r
    assert _inject(fa, 1, run) == 0          # other kernels' modes leave the quantizer alone
    bits_set = _inject(fa, 5, run)
    assert bits_set == 1 << 16, "the quantizer should report bit 16 (bits=%#x)" % bits_set
    x8, desc = run()
    assert fa.fa_device_status() == 0
    ref8, ref_desc = fp8_quantize(bf16_bits_to_f32(bits), None)
    assert np.array_equal(x8.cpu().numpy(), ref8) and np.array_equal(desc.cpu().numpy(), ref_desc)
