"""Failure detection without a GPU fault: a copy that never arrives makes the
kernel's bounded waits run out; the kernel must report it in the device
status word, exit cleanly and leave the context usable."""
import numpy as np
import pytest
import torch

from fa_inputs import make_dense
from fa_testutil import run_gpu, oracle_full, compare


def test_hook_argument_checks():
    import exact_attention_42_gb300 as fa
    fa.build()
    with pytest.raises(fa.FaError):
        fa.fa_debug_fault_injection(2, 0.1)
    with pytest.raises(fa.FaError):
        fa.fa_debug_fault_injection(1, 11.0)
    fa.fa_debug_fault_injection(0, 0.0)


@pytest.mark.gpu
def test_withheld_copy_times_out_and_context_survives():
    import exact_attention_42_gb300 as fa
    fa.build()
    dev = torch.device("cuda", 0)
    prob = make_dense(1, 4, 4, 512, 512, 64, seed=17, causal=True)
    fa.fa_device_status()
    fa.fa_debug_fault_injection(1, 0.05)
    try:
        run_gpu(fa, prob, dev)           # returns once the kernel has given up and exited
    finally:
        fa.fa_debug_fault_injection(0, 0.0)
    bits = fa.fa_device_status()
    # Whichever role's bounded wait ran out first raised the abort: the K/V
    # producer (bit 0, its slot is never released) or the MMA issuer (bit 1,
    # the copy never lands).  Roles that then saw the abort flag leave quietly.
    assert bits & 0b11, "a bounded wait should have run out (bits=%#x)" % bits
    # The same process keeps working.
    o, lse = run_gpu(fa, prob, dev)
    ref_o, ref_lse = oracle_full(prob)
    compare(o, lse, ref_o, ref_lse, "after fault injection")
    assert fa.fa_device_status() == 0
