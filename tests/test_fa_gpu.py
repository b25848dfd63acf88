"""GPU parity: the tcgen05 kernel, called through the C ABI, against the fp64
CPU oracle on the same seeded bf16 inputs.

Tolerances: max |O - O_ref| <= 2e-2 and |LSE - LSE_ref| <= 1e-3 * max(1, |LSE_ref|)
(bf16 inputs, fp32 accumulation).  Every workload, the full-size ones
included, is compared element by element, in the same launch configuration
the bench uses; the full-size ones head by head, so that the oracle's memory
stays bounded.
"""
import math

import numpy as np
import pytest
import torch

from fa_inputs import make_dense, make_varlen, make_workload, f64_to_bf16_bits, WORKLOADS
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


# ---------------------------------------------------------------- workloads

@pytest.mark.parametrize("name", ["tiny_b1_h2_n128_d64", "b4_h16_n1024_d64", "b4_h16_n1024_d64_causal"])
def test_workload_full(fa, dev, name):
    prob = make_workload(name)
    o, lse = run_gpu(fa, prob, dev)
    ref_o, ref_lse = oracle_full(prob)
    compare(o, lse, ref_o, ref_lse, name)


FULL_SIZE = ["b2_h32_n4096_d128_causal", "gqa_b1_hq32_hkv8_n16384_d128_causal", "varlen16_h16_d128_causal"]


@pytest.mark.parametrize("name", FULL_SIZE)
def test_workload_full_size(fa, dev, name):
    """The full-size workloads, every element of O and LSE against the oracle."""
    prob = make_workload(name)
    o, lse = run_gpu(fa, prob, dev, keep_on_device=True)
    compare_per_head(o, lse, prob)


# ------------------------------------------------------------- edge shapes

EDGE = [
    # (B, Hq, Hkv, Nq, Nk, d, causal)
    (2, 3, 3, 200, 200, 128, True),     # ragged tail, several tiles
    (2, 3, 3, 200, 200, 128, False),
    (1, 2, 1, 77, 300, 64, True),       # Nq < Nk: bottom-right diagonal
    (1, 2, 2, 300, 77, 64, True),       # Nq > Nk: first rows see no key
    (1, 2, 2, 300, 77, 128, False),
    (1, 1, 1, 5, 5, 64, True),          # shorter than one tile
    (1, 1, 1, 1, 1, 128, False),
    (1, 1, 1, 1, 700, 128, True),       # one query row against many keys
    (1, 32, 1, 130, 130, 128, True),    # MQA: 32 query heads on one KV head
    (2, 8, 2, 257, 257, 64, True),      # GQA g=4, tile + 1 row
    (1, 4, 4, 512, 512, 128, True),     # exact multiple of the 256-row unit
    (3, 5, 5, 384, 640, 64, False),
]


@pytest.mark.parametrize("shape", EDGE, ids=["-".join(map(str, s)) for s in EDGE])
def test_edge_shapes(fa, dev, shape):
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    prob = make_dense(B, Hq, Hkv, Nq, Nk, d, seed=sum(shape), causal=causal, name="edge")
    o, lse = run_gpu(fa, prob, dev)
    ref_o, ref_lse = oracle_full(prob)
    compare(o, lse, ref_o, ref_lse, str(shape))


# More units than SMs: the host-built worker lists (SchedTable) run them.
SCHEDULED = [
    (3, 20, 5, 1000, 1300, 128, True),   # GQA, Nq < Nk, ragged
    (2, 40, 40, 700, 700, 64, False),
    (2, 24, 8, 1500, 900, 128, True),    # Nq > Nk: early rows see no key
]


@pytest.mark.parametrize("shape", SCHEDULED, ids=["-".join(map(str, s)) for s in SCHEDULED])
def test_scheduled_shapes(fa, dev, shape):
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    assert fa.fa_debug_schedule(0, B, Hq, Hkv, Nq, Nk, d, causal, torch.cuda.get_device_properties(dev)
                                .multi_processor_count) is not None
    prob = make_dense(B, Hq, Hkv, Nq, Nk, d, seed=sum(shape) + 11, causal=causal, name="scheduled")
    o, lse = run_gpu(fa, prob, dev, keep_on_device=True)
    compare_per_head(o, lse, prob)


VARLEN = [
    ([1, 127, 128, 129, 0, 300, 256, 257], 4, 2, 64, True),
    ([1, 127, 128, 129, 0, 300, 256, 257], 4, 2, 128, False),
    ([513, 3, 1000], 2, 2, 128, True),
    ([0, 0, 64], 1, 1, 64, True),
]


@pytest.mark.parametrize("case", VARLEN, ids=["v%d" % i for i in range(len(VARLEN))])
def test_varlen(fa, dev, case):
    lens, Hq, Hkv, d, causal = case
    prob = make_varlen(lens, Hq, Hkv, d, seed=len(lens) + d, causal=causal)
    o, lse = run_gpu(fa, prob, dev)
    ref_o, ref_lse = oracle_full(prob)
    compare(o, lse, ref_o, ref_lse, "varlen %s" % lens)


def test_no_keys(fa, dev):
    prob = make_dense(1, 2, 2, 100, 0, 64, seed=3, causal=False)
    o, lse = run_gpu(fa, prob, dev)
    assert np.all(o == 0.0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("d", [64, 128])
def test_growing_scores_force_rescales(fa, dev, d):
    """Scores that grow along the key axis move the running max by more than
    the rescale threshold in every K/V tile (exercises the O correction; at
    d = 64 the correction first waits for the tile's previous P V product,
    which runs behind the next QK there)."""
    N = 1024
    # s_j = scale * 0.25 * d * k_j grows by about 20 (d = 128) or 14 (d = 64)
    # log2 units per 128-key tile.
    q = np.full((1, 2, N, d), 0.25)
    ramp = np.linspace(0.0, 40.0, N)[None, None, :, None]
    k = np.broadcast_to(ramp, (1, 2, N, d)) + 0.01 * np.random.default_rng(0).standard_normal((1, 2, N, d))
    v = np.random.default_rng(1).standard_normal((1, 2, N, d))
    for causal in (False, True):
        prob = make_dense(1, 2, 2, N, N, d, seed=0, causal=causal)
        prob.q, prob.k, prob.v = (f64_to_bf16_bits(x) for x in (q, k, v))
        prob.scale = 1.0 / math.sqrt(d)
        o, lse = run_gpu(fa, prob, dev)
        ref_o, ref_lse = oracle_full(prob)
        compare(o, lse, ref_o, ref_lse, "growing scores causal=%s" % causal)


def test_large_score_magnitudes(fa, dev):
    """Scores spanning hundreds of units (exp would overflow without the max)."""
    prob = make_dense(1, 2, 2, 300, 300, 64, seed=21, causal=True)
    prob.scale = 4.0
    o, lse = run_gpu(fa, prob, dev)
    ref_o, ref_lse = oracle_full(prob)
    assert np.max(np.abs(ref_lse)) > 50
    compare(o, lse, ref_o, ref_lse, "large scores")


# ------------------------------------------------------------- properties

def test_deterministic_and_stream(fa, dev):
    prob = make_dense(2, 4, 2, 600, 600, 128, seed=5, causal=True)
    q, k, v = (to_dev(x, dev) for x in (prob.q, prob.k, prob.v))
    o1, l1 = fa.fwd(q, k, v, causal=True)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        o2, l2 = fa.fwd(q, k, v, causal=True)
    s.synchronize()
    torch.cuda.synchronize(dev)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_output_canaries(fa, dev):
    """Writes stay inside O and LSE (guard regions around both are untouched)."""
    lens = [1, 130, 0, 255, 257]
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
    compare(o.float().cpu().numpy().astype(np.float64), l.cpu().numpy().astype(np.float64), ref_o, ref_lse, "canary")


def test_misaligned_pointer_is_rejected(fa, dev):
    buf = torch.zeros(1 * 1 * 64 * 64 + 8, dtype=torch.bfloat16, device=dev)
    q = buf[1:1 + 64 * 64].view(1, 1, 64, 64)
    k = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16, device=dev)
    with pytest.raises(fa.FaError) as e:
        fa.fwd(q, k, k)
    assert e.value.status == 3


def test_host_entry_matches_device_entry(fa, dev):
    prob = make_dense(1, 4, 4, 256, 256, 64, seed=13, causal=True)
    qh, kh, vh = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in (prob.q, prob.k, prob.v))
    o_h, l_h = fa.fwd_host(qh, kh, vh, causal=True)
    o_d, l_d = fa.fwd(qh.to(dev), kh.to(dev), vh.to(dev), causal=True)
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())


@pytest.mark.parametrize("chunks", [1, 3, 7])
def test_host_entry_pieces_gqa(fa, dev, chunks):
    # fa_fwd_host cuts a dense problem into (batch, key/value head range)
    # slices; uneven slices must give the device entry's result bit for bit.
    prob = make_dense(2, 12, 3, 300, 500, 128, seed=14, causal=True)
    qh, kh, vh = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in (prob.q, prob.k, prob.v))
    o_h, l_h = fa.fwd_host(qh, kh, vh, causal=True, chunks=chunks)
    o_d, l_d = fa.fwd(qh.to(dev), kh.to(dev), vh.to(dev), causal=True)
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())


@pytest.mark.parametrize("chunks", [1, 3])
@pytest.mark.parametrize("shape", [(2, 16, 4, 1, 3000, 128), (1, 32, 8, 4, 2500, 64)],
                         ids=["q1-gqa4-d128", "q4-gqa4-d64"])
def test_host_entry_decode_shapes(fa, dev, shape, chunks):
    # Few query rows per key/value head (R = group * Nq <= 16): every piece
    # goes to the split-KV kernel, and every element is checked against the
    # oracle.  The split count follows the number of (batch, key/value head)
    # groups in a launch; with at most 8 groups here the whole problem and
    # every piece take the same splits, so the pieces also match the device
    # entry bit for bit (with many groups they would not, in the last bits).
    B, Hq, Hkv, Nq, Nk, d = shape
    prob = make_dense(B, Hq, Hkv, Nq, Nk, d, seed=16 + Nq, causal=False)
    qh, kh, vh = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in (prob.q, prob.k, prob.v))
    o_h, l_h = fa.fwd_host(qh, kh, vh, causal=False, chunks=chunks)
    o_d, l_d = fa.fwd(qh.to(dev), kh.to(dev), vh.to(dev), causal=False)
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())
    ref_o, ref_lse = oracle_full(prob)
    compare(o_h.float().numpy().astype(np.float64), l_h.numpy().astype(np.float64), ref_o, ref_lse, "decode host")


@pytest.mark.parametrize("chunks", [2, 5])
def test_host_entry_d64_pieces(fa, dev, chunks):
    # d = 64, non-causal, Nq != Nk, uneven pieces: the device entry's result
    # bit for bit, and every element against the oracle.
    prob = make_dense(3, 10, 5, 333, 190, 64, seed=17, causal=False)
    qh, kh, vh = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in (prob.q, prob.k, prob.v))
    o_h, l_h = fa.fwd_host(qh, kh, vh, causal=False, chunks=chunks)
    o_d, l_d = fa.fwd(qh.to(dev), kh.to(dev), vh.to(dev), causal=False)
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())
    ref_o, ref_lse = oracle_full(prob)
    compare(o_h.float().numpy().astype(np.float64), l_h.numpy().astype(np.float64), ref_o, ref_lse, "d64 host")


def test_host_entry_no_keys(fa, dev):
    # Nk = 0: no copies of K and V, O = 0 and LSE = -inf for every row.
    q = torch.randn(2, 4, 70, 128).to(torch.bfloat16).pin_memory()
    k = torch.empty(2, 2, 0, 128, dtype=torch.bfloat16).pin_memory()
    o_h, l_h = fa.fwd_host(q, k, k.clone(), causal=False, chunks=3)
    assert torch.all(o_h == 0) and torch.all(torch.isneginf(l_h))


def test_host_entry_packed(fa, dev):
    prob = make_varlen([5, 300, 129, 0, 64], 4, 2, 64, seed=15, causal=True)
    qh, kh, vh = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in (prob.q, prob.k, prob.v))
    cu = torch.from_numpy(prob.cu_seqlens)
    o_h, l_h = fa.fwd_host(qh, kh, vh, causal=True, cu_seqlens=cu)
    o_d, l_d = fa.fwd(qh.to(dev), kh.to(dev), vh.to(dev), causal=True, cu_seqlens=cu.to(dev))
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())
    ref_o, ref_lse = oracle_full(prob)
    compare(o_h.float().numpy().astype(np.float64), l_h.numpy().astype(np.float64), ref_o, ref_lse, "packed host")


def test_software_exp2_error_bound(fa, dev):
    """The FMA-pipe 2^x used for part of the exponentials: relative error below
    the minimax bound of its polynomial (7.5e-5, a little slack for rounding)."""
    x = torch.cat([torch.linspace(-125.0, 8.0, 1 << 20, dtype=torch.float32),
                   torch.tensor([0.0, 0.5, -0.5, 1.0, -1.0, 7.75, -124.5, -125.0], dtype=torch.float32)]).to(dev)
    y = torch.empty_like(x)
    fa.fa_debug_exp2_soft(x.data_ptr(), y.data_ptr(), x.numel(), torch.cuda.current_stream(dev).cuda_stream)
    torch.cuda.synchronize(dev)
    xe = x.double().cpu()
    rel = ((y.double().cpu() - torch.exp2(xe)) / torch.exp2(xe)).abs()
    assert float(rel.max()) < 8e-5, float(rel.max())
    # Arguments below the clamp stay tiny and positive (never wrap negative or to inf).
    z = torch.tensor([-126.0, -300.0, -1e30], dtype=torch.float32, device=dev)
    w = torch.empty_like(z)
    fa.fa_debug_exp2_soft(z.data_ptr(), w.data_ptr(), 3, torch.cuda.current_stream(dev).cuda_stream)
    torch.cuda.synchronize(dev)
    assert bool(((w > 0) & (w < 1e-37)).all())


def test_dependent_calls_in_one_stream(fa, dev):
    """Each launch may start before the previous kernel in its stream has
    finished and must wait for it before touching global memory: a chain of
    calls that read one another's outputs, issued back to back, gives
    bitwise the same results as the same chain with a synchronisation after
    every call (the kernels are deterministic)."""
    prob = make_dense(2, 8, 8, 2048, 2048, 128, seed=31, causal=True)
    q, k, v = (to_dev(x, dev) for x in (prob.q, prob.k, prob.v))
    small = make_dense(1, 2, 2, 300, 300, 64, seed=32, causal=False)
    qs, ks, vs = (to_dev(x, dev) for x in (small.q, small.k, small.v))

    def chain(sync):
        outs = []
        o1, l1 = fa.fwd(q, k, v, causal=True)
        outs += [o1, l1]
        if sync:
            torch.cuda.synchronize(dev)
        o2, l2 = fa.fwd(o1, k, v, causal=True)           # reads the first call's O as queries
        outs += [o2, l2]
        if sync:
            torch.cuda.synchronize(dev)
        o3, l3 = fa.fwd(qs, ks, vs)                        # a short launch between long ones
        outs += [o3, l3]
        o4, l4 = fa.fwd(q, o2, o1, causal=False)          # reads both earlier outputs as K and V
        outs += [o4, l4]
        if sync:
            torch.cuda.synchronize(dev)
        torch.cuda.synchronize(dev)
        return outs

    a = chain(False)
    b = chain(True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    ref_o, ref_lse = oracle_full(prob)
    compare(a[0].float().cpu().numpy().astype(np.float64), a[1].cpu().numpy().astype(np.float64), ref_o, ref_lse,
            "first call of the chain")
