"""Shared helpers for the GPU parity tests (test code only)."""
import numpy as np
import torch

from fa_inputs import bf16_bits_to_f64
from oracle import attention_fwd, attention_rows

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


def sample_rows(prob, n, seed):
    """(b or seq, h, i) samples covering first/last rows, tile edges and random rows."""
    rng = np.random.default_rng(seed)
    out = []
    seqs = prob.seqlens()
    for _ in range(n):
        b = int(rng.integers(prob.B))
        while seqs[b] == 0:
            b = int(rng.integers(prob.B))
        h = int(rng.integers(prob.Hq))
        L = seqs[b]
        pick = rng.integers(6)
        i = [0, L - 1, min(L - 1, 127), min(L - 1, 128), min(L - 1, 255), int(rng.integers(L))][pick]
        out.append((b, h, int(i)))
    return out


def compare_sampled(o, lse, prob, samples):
    q, k, v = (bf16_bits_to_f64(x) for x in (prob.q, prob.k, prob.v))
    ref_o, ref_lse = attention_rows(q, k, v, prob.scale, prob.causal, samples, cu_seqlens=prob.cu_seqlens)
    if prob.cu_seqlens is None:
        idx = [(b, h, i) for b, h, i in samples]
    else:
        cu = prob.cu_seqlens
        idx = [(h, int(cu[s]) + i) for s, h, i in samples]
    got_o = np.stack([np.asarray(o[ix].float().cpu() if torch.is_tensor(o) else o[ix], dtype=np.float64)
                      for ix in idx])
    got_l = np.array([float(lse[ix]) for ix in idx], dtype=np.float64)
    return compare(got_o, got_l, ref_o, ref_lse, prob.name + " (sampled)")
