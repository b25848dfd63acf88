"""Host-side work schedules of the persistent kernels (fa_debug_schedule).

The kernels' units are blocks of query rows (forward, backward dQ) or of keys
(backward dK/dV) of one head.  For dense problems the host hands each
persistent CTA a list of units: heads are taken in groups whose K/V (or Q/dO)
tiles fit in L2, the longest units first, each to the worker predicted to be
free first.  These checks need no GPU: every unit is run exactly once, the
predicted busiest worker stays within list scheduling's bound (mean load +
the longest unit, Graham 1969), and concurrent units span few heads.  The
unit costs are derived here again from the geometry of the mask.
"""
import pytest

import exact_attention_42_gb300 as fa

SMS = 152
L2_GROUP_BYTES = 32 * 2 ** 20


@pytest.fixture(scope="module", autouse=True)
def _built():
    fa.build()


def fwd_units(B, Hq, Hkv, Nq, Nk, causal, rows=256, tile=128):
    """(cost in K/V steps, KV head) of every forward unit, in the kernel's unit order."""
    nqb = -(-Nq // rows)
    out = []
    for u in range(B * Hq * nqb):
        qb, bh = nqb - 1 - u // (B * Hq), u % (B * Hq)
        steps = 0
        for t in range(rows // tile):
            q0 = qb * rows + t * tile
            if q0 >= Nq or Nk == 0:
                continue
            last = Nk - 1
            if causal:
                last = min(last, min(q0 + tile - 1, Nq - 1) + Nk - Nq)
            if last >= 0:
                steps = max(steps, last // 128 + 1)
        out.append((steps + 2, (bh // Hq) * Hkv + (bh % Hq) // (Hq // Hkv)))
    return out


def bwd_units(B, Hq, Hkv, Nq, Nk, causal, kv, tile=128):
    nqt, nkt, g = -(-Nq // tile), -(-Nk // tile), Hq // Hkv
    out = []
    if not kv:
        for u in range(B * Hq * nqt):
            q0, bh = (nqt - 1 - u // (B * Hq)) * tile, u % (B * Hq)
            last = Nk - 1
            if causal:
                last = min(last, min(q0 + tile - 1, Nq - 1) + Nk - Nq)
            steps = last // tile + 1 if (q0 < Nq and last >= 0) else 0
            out.append((steps + 1, (bh // Hq) * Hkv + (bh % Hq) // g))
    else:
        for u in range(B * Hkv * nkt):
            key0, bkv = (u // (B * Hkv)) * tile, u % (B * Hkv)
            first = 0
            if causal:
                qmin = key0 - (Nk - Nq)
                first = 0 if qmin <= 0 else (nqt if qmin >= Nq else qmin // tile)
            out.append((g * (nqt - first) + 1, bkv))
    return out


def simulate(lists, units):
    """Predicted finish time per worker and the KV heads running at sampled times."""
    spans, ends = [], []
    for lst in lists:
        t = 0.0
        for u in lst:
            c, head = units[u]
            spans.append((t, t + c, head))
            t += c
        ends.append(t)
    T = max(ends)
    heads = [len({h for a, b, h in spans if a <= T * i / 64 < b}) for i in range(1, 64)]
    return ends, max(heads)


CASES = [
    # kernel, (B, Hq, Hkv, Nq, Nk, d, causal)
    (0, (2, 32, 32, 4096, 4096, 128, True)),
    (0, (1, 32, 8, 16384, 16384, 128, True)),
    (0, (4, 16, 16, 1024, 1024, 64, False)),
    (0, (4, 16, 16, 1024, 1024, 64, True)),
    (0, (3, 20, 5, 1000, 1300, 128, True)),
    (2, (2, 32, 32, 4096, 4096, 128, True)),
    (3, (2, 32, 32, 4096, 4096, 128, True)),
    (2, (1, 32, 8, 16384, 16384, 128, True)),
    (3, (1, 32, 8, 16384, 16384, 128, True)),
    (3, (2, 16, 16, 1300, 1300, 64, True)),
]


@pytest.mark.parametrize("kernel,shape", CASES, ids=["k%d-%s" % (k, "-".join(map(str, s))) for k, s in CASES])
def test_schedule_covers_every_unit_and_balances(kernel, shape):
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    units = (fwd_units(B, Hq, Hkv, Nq, Nk, causal) if kernel < 2
             else bwd_units(B, Hq, Hkv, Nq, Nk, causal, kv=kernel == 3))
    lists = fa.fa_debug_schedule(kernel, B, Hq, Hkv, Nq, Nk, d, causal, SMS)
    assert lists is not None and len(lists) == min(SMS, len(units))
    flat = sorted(u for lst in lists for u in lst)
    assert flat == list(range(len(units))), "every unit exactly once"
    ends, _ = simulate(lists, units)
    mean = sum(c for c, _ in units) / len(lists)
    longest = max(c for c, _ in units)
    assert max(ends) <= mean + longest + 1e-6, "list scheduling bound"


def test_headline_schedule_keeps_few_heads_in_flight():
    # The built-in snake order starts the longest unit of all 64 heads at once
    # (134 MB of K/V, more than L2); the table keeps the concurrent units
    # within about two groups of 16 heads (2 MB of K/V each).
    B, Hq, Hkv, Nq, Nk, d, causal = 2, 32, 32, 4096, 4096, 128, True
    units = fwd_units(B, Hq, Hkv, Nq, Nk, causal)
    lists = fa.fa_debug_schedule(0, B, Hq, Hkv, Nq, Nk, d, causal, SMS)
    ends, heads = simulate(lists, units)
    group = L2_GROUP_BYTES // (2 * Nk * d * 2)
    assert group == 16
    assert heads <= 2 * group, heads
    mean = sum(c for c, _ in units) / len(lists)
    assert max(ends) <= 1.02 * mean


def test_no_table_when_units_fit_one_round_or_for_unknown_kernel():
    assert fa.fa_debug_schedule(0, 1, 2, 2, 128, 128, 64, True, SMS) is None
    assert fa.fa_debug_schedule(1, 2, 32, 32, 4096, 4096, 128, True, SMS) is None   # the 8-bit path: snake order
    assert fa.fa_debug_schedule(2, 1, 4, 4, 1024, 1024, 128, True, SMS) is None   # 32 units
    with pytest.raises(fa.FaError):
        fa.fa_debug_schedule(4, 1, 2, 2, 128, 128, 64, True, SMS)
    with pytest.raises(fa.FaError):
        fa.fa_debug_schedule(0, 1, 3, 2, 128, 128, 64, True, SMS)   # Hq not a multiple of Hkv
