"""The C ABI's launches inside CUDA graphs: a forward, a backward, an e4m3
quantization and an 8-bit forward captured into one graph and replayed
must give the eager calls' results bit for bit, with a clean device status.
(Every launch carries the programmatic-serialization attribute and the
forward's work lists ride in its kernel parameters, so a captured launch
owns everything it needs.)"""
import numpy as np
import pytest
import torch

from fa_inputs import make_dense, make_dout
from fa_testutil import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_42_gb300 as m
    m.build()
    m.lib()
    return m


def test_captured_calls_replay_bit_for_bit(fa):
    dev = torch.device("cuda", 0)
    prob = make_dense(2, 6, 3, 700, 912, 128, seed=61, causal=True)   # more units than SMs: work lists
    q, k, v, do = (to_dev(x, dev) for x in (prob.q, prob.k, prob.v, make_dout(prob, 62)))
    fa.fa_device_status()

    def calls(out):
        o, lse = fa.fwd(q, k, v, causal=True, scale=prob.scale, out=out["o"], lse=out["lse"])
        fa.bwd(q, k, v, o, lse, do, causal=True, scale=prob.scale, dq=out["dq"], dk=out["dk"], dv=out["dv"],
               delta=out["delta"])
        q8, qd = fa.fp8_quantize(q, None, out=out["q8"], descale=out["qd"])
        k8, kd = fa.fp8_quantize(k, None, out=out["k8"], descale=out["kd"])
        vt8, vd = fa.fp8_quantize(v, None, transpose=True, out=out["vt8"], descale=out["vd"])
        fa.fwd_fp8(q8, k8, vt8, qd, kd, vd, causal=True, scale=prob.scale, out=out["o8"], lse=out["lse8"])

    def buffers():
        f32 = dict(dtype=torch.float32, device=dev)
        u8 = dict(dtype=torch.uint8, device=dev)
        return {"o": torch.empty_like(q), "lse": torch.empty(q.shape[:-1], **f32),
                "dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
                "delta": torch.empty(q.shape[:-1], **f32),
                "q8": torch.empty(q.shape, **u8), "qd": torch.empty(q.shape[:2], **f32),
                "k8": torch.empty(k.shape, **u8), "kd": torch.empty(k.shape[:2], **f32),
                "vt8": torch.empty(v.shape[:2] + (v.shape[3], v.shape[2]), **u8), "vd": torch.empty(v.shape[:2], **f32),
                "o8": torch.empty_like(q), "lse8": torch.empty(q.shape[:-1], **f32)}

    eager = buffers()
    calls(eager)
    torch.cuda.synchronize(dev)
    assert fa.fa_device_status() == 0

    graphed = buffers()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):          # warm-up outside the capture (one-time set-up)
        calls(graphed)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    for t in graphed.values():
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        calls(graphed)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize(dev)
    assert fa.fa_device_status() == 0
    for name in eager:
        assert torch.equal(graphed[name], eager[name]), name
    assert bool(torch.isfinite(graphed["o8"].float()).all())
    assert np.isfinite(graphed["dq"].float().cpu().numpy()).all()
