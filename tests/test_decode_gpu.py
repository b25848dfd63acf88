"""GPU parity of the split-KV decode path (few query rows per key/value head)
against the fp64 oracle, through fa_decode and through fa_fwd's dispatch."""
import numpy as np
import pytest
import torch

from fa_inputs import make_dense, make_workload
from fa_testutil import run_gpu, oracle_full, compare, compare_per_head, to_dev

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


DECODE = [
    # (B, Hq, Hkv, Nq, Nk, d, causal)
    (2, 8, 2, 1, 3000, 128, False),     # GQA g=4, one token
    (3, 8, 2, 4, 2049, 128, True),      # 4 tokens, bottom-right causal, ragged key count
    (1, 16, 1, 1, 777, 64, False),      # MQA g=16
    (2, 4, 4, 16, 5000, 128, True),     # no GQA, 16 tokens
    (1, 2, 2, 3, 40, 64, True),         # fewer keys than one tile
    (2, 8, 8, 2, 65, 128, False),       # one key past a tile
    (1, 32, 8, 4, 12000, 128, True),    # R = 16 rows per key/value head, many splits
    (4, 4, 1, 2, 1, 128, True),         # a single key
]


def _run_decode(fa, prob, dev):
    q, k, v = (to_dev(x, dev) for x in (prob.q, prob.k, prob.v))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=dev)
    st = fa.fa_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), prob.B, prob.Hq,
                      prob.Hkv, prob.Nq, prob.Nk, prob.d, prob.scale, int(prob.causal),
                      torch.cuda.current_stream(dev).cuda_stream)
    assert st == 0, fa.fa_status_string(st)
    torch.cuda.synchronize(dev)
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("shape", DECODE, ids=["-".join(map(str, s)) for s in DECODE])
def test_decode_matches_oracle(fa, dev, shape):
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    prob = make_dense(B, Hq, Hkv, Nq, Nk, d, seed=sum(shape) + 100, causal=causal, name="decode")
    ref_o, ref_lse = oracle_full(prob)
    o, lse = _run_decode(fa, prob, dev)
    compare(o, lse, ref_o, ref_lse, "fa_decode %s" % (shape,))
    o2, lse2 = run_gpu(fa, prob, dev)          # fa_fwd dispatches the same shapes here
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_decode_rejects_large_groups(fa, dev):
    q = torch.zeros(1, 32, 1, 128, dtype=torch.bfloat16, device=dev)   # g = 32 > 16 rows
    k = torch.zeros(1, 1, 64, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(1, 32, 1, dtype=torch.float32, device=dev)
    st = fa.fa_decode(q.data_ptr(), k.data_ptr(), k.data_ptr(), q.data_ptr(), lse.data_ptr(), 1, 32, 1, 1, 64, 128,
                      0.1, 0, 0)
    assert st == 4


@pytest.mark.parametrize("name", ["decode_b8_hq32_hkv8_nq1_nk32768_d128", "decode_b16_hq32_hkv8_nq4_nk8192_d128_causal"])
def test_decode_workloads_full_size(fa, dev, name):
    """The full-size decode workloads, every element against the oracle."""
    prob = make_workload(name)
    o, lse = run_gpu(fa, prob, dev, keep_on_device=True)
    compare_per_head(o, lse, prob)
