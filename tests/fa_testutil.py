"""Shared helpers for the GPU parity tests (test code only)."""
import numpy as np
import torch

from fa_inputs import bf16_bits_to_f64
from oracle import attention_fwd

O_ATOL = 2e-2     # max |O_gpu - O_ref| for bf16 inputs, fp32 accumulation
LSE_RTOL = 1e-3   # |LSE_gpu - LSE_ref| <= LSE_RTOL * max(1, |LSE_ref|)


def to_dev(bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def run_gpu(fa, prob, dev, keep_on_device=False):
    q, k, v = to_dev(prob.q, dev), to_dev(prob.k, dev), to_dev(prob.v, dev)
    cu = None if prob.cu_seqlens is None else torch.from_numpy(prob.cu_seqlens).to(dev)
    o, lse = fa.fwd(q, k, v, causal=prob.causal, scale=prob.scale, cu_seqlens=cu)
    torch.cuda.synchronize(dev)
    if keep_on_device:
        return o, lse
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def oracle_full(prob):
    q, k, v = (bf16_bits_to_f64(x) for x in (prob.q, prob.k, prob.v))
    return attention_fwd(q, k, v, prob.scale, prob.causal, cu_seqlens=prob.cu_seqlens)


def compare(o, lse, ref_o, ref_lse, what=""):
    """Element-wise check; -inf LSE (rows with no visible key) must match exactly."""
    assert o.shape == ref_o.shape and lse.shape == ref_lse.shape
    assert np.all(np.isfinite(o)), what + ": non-finite O"
    inf_ref = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), inf_ref), what + ": -inf LSE pattern differs"
    assert np.all(o[inf_ref] == 0.0), what + ": fully masked rows must be 0"
    err_o = float(np.max(np.abs(o - ref_o))) if o.size else 0.0
    fin = ~inf_ref
    err_l = float(np.max(np.abs(lse[fin] - ref_lse[fin]) / np.maximum(1.0, np.abs(ref_lse[fin])))) if fin.any() else 0.0
    assert err_o <= O_ATOL, "%s: max|dO| = %.4g" % (what, err_o)
    assert err_l <= LSE_RTOL, "%s: max rel dLSE = %.4g" % (what, err_l)
    return err_o, err_l


def compare_per_head(o, lse, prob, what=None):
    """Every element of a device result (O, LSE) against the oracle, one
    (batch, head) or (head, packed batch) slice at a time, so that host memory
    stays bounded at full size.  Returns the largest errors seen."""
    what = what or prob.name
    f64 = bf16_bits_to_f64
    g = prob.Hq // prob.Hkv
    worst_o = worst_l = 0.0
    if prob.cu_seqlens is None:
        for b in range(prob.B):
            for h in range(prob.Hq):
                kvh = h // g
                ref_o, ref_l = attention_fwd(f64(prob.q[b:b + 1, h:h + 1]), f64(prob.k[b:b + 1, kvh:kvh + 1]),
                                             f64(prob.v[b:b + 1, kvh:kvh + 1]), prob.scale, prob.causal)
                got_o = o[b:b + 1, h:h + 1].float().cpu().numpy().astype(np.float64)
                got_l = lse[b:b + 1, h:h + 1].cpu().numpy().astype(np.float64)
                eo, el = compare(got_o, got_l, ref_o, ref_l, "%s b=%d h=%d" % (what, b, h))
                worst_o, worst_l = max(worst_o, eo), max(worst_l, el)
    else:
        for h in range(prob.Hq):
            kvh = h // g
            ref_o, ref_l = attention_fwd(f64(prob.q[h:h + 1]), f64(prob.k[kvh:kvh + 1]), f64(prob.v[kvh:kvh + 1]),
                                         prob.scale, prob.causal, cu_seqlens=prob.cu_seqlens)
            got_o = o[h:h + 1].float().cpu().numpy().astype(np.float64)
            got_l = lse[h:h + 1].cpu().numpy().astype(np.float64)
            eo, el = compare(got_o, got_l, ref_o, ref_l, "%s h=%d" % (what, h))
            worst_o, worst_l = max(worst_o, eo), max(worst_l, el)
    return worst_o, worst_l
