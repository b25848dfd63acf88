"""Pins for the fp64 oracle (CPU only).

The oracle is the plain definition of attention ("FlashAttention面试讲解"
canvas, ``std-text``).  These tests tie it to things other than itself:
hand-derived values for the canvas's two-tile exercise, closed forms (Q = 0,
constant V), invariants (rows of P sum to 1, shift invariance, permutation
equivariance), brute force with pure-Python loops on tiny inputs, a library
routine (torch's scaled_dot_product_attention in float64), and a separately
written online-softmax recurrence (canvas ``formula-text`` / ``qa2-a``).
``test_planted_mistakes_are_caught`` plants plausible mistakes in copies of
the oracle and checks that every one of them fails at least one pin.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle.attention as oa
from oracle import attention_fwd, attention_rows
from fa_inputs import make_dense, make_varlen, bf16_bits_to_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "two_tile_worked.json")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# --------------------------------------------------------------------------
# Pin checks, written against any oracle-like callable ``fwd`` so that the
# planted-mistake test can run them against broken copies.
# --------------------------------------------------------------------------

def _golden_case():
    with open(GOLDEN) as f:
        g = json.load(f)
    q = np.array(g["q"], dtype=np.float64)[None, None]
    k = np.log(np.array(g["k_exp"], dtype=np.float64))[None, None]
    v = np.array(g["v"], dtype=np.float64)[None, None]
    return g, q, k, v


def pin_golden(fwd):
    g, q, k, v = _golden_case()
    for mode, causal in (("noncausal", False), ("causal", True)):
        o, lse = fwd(q, k, v, 1.0, causal)
        want_o = np.array([[float(Fraction(n, d)) for n, d in row] for row in g[mode]["O"]])
        want_lse = np.log(np.array(g[mode]["LSE_exp"], dtype=np.float64))
        np.testing.assert_allclose(o[0, 0], want_o, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[0, 0], want_lse, rtol=0, atol=1e-13)


def pin_p_rows_sum_to_one(fwd_p):
    for causal, nq, nk in ((False, 7, 9), (True, 7, 9), (True, 9, 6)):
        q, k, v = _rand((1, 2, nq, 4), 1), _rand((1, 2, nk, 4), 2), _rand((1, 2, nk, 4), 3)
        _, lse, p = fwd_p(q, k, v, 0.5, causal)
        sums = p.sum(axis=-1)
        has = np.isfinite(lse)
        assert np.all(np.abs(sums[has] - 1.0) <= 1e-12)
        assert np.all(sums[~has] == 0.0)


def pin_zero_q_mean_of_v(fwd):
    # Q = 0 makes every score 0: O is the mean of V over the valid keys and
    # LSE = ln(number of valid keys).  Causal masks are bottom-right aligned.
    for causal, nq, nk in ((False, 5, 11), (True, 5, 11), (True, 11, 5), (True, 8, 8)):
        q = np.zeros((2, 2, nq, 3))
        k, v = _rand((2, 2, nk, 3), 4), _rand((2, 2, nk, 3), 5)
        o, lse = fwd(q, k, v, 0.7, causal)
        for i in range(nq):
            nvalid = min(nk, i + (nk - nq) + 1) if causal else nk
            if nvalid <= 0:
                assert np.all(o[:, :, i] == 0.0) and np.all(lse[:, :, i] == -np.inf)
                continue
            np.testing.assert_allclose(o[:, :, i], v[:, :, :nvalid].mean(axis=2), rtol=0, atol=1e-13)
            np.testing.assert_allclose(lse[:, :, i], math.log(nvalid), rtol=0, atol=1e-13)


def pin_constant_v(fwd):
    for causal in (False, True):
        q, k = _rand((1, 3, 6, 4), 6), _rand((1, 3, 6, 4), 7)
        c = np.array([1.5, -2.0, 0.25, 3.0])
        v = np.broadcast_to(c, (1, 3, 6, 4)).copy()
        o, _ = fwd(q, k, v, 0.9, causal)
        np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=0, atol=1e-13)


def pin_brute_force(fwd):
    # Pure-Python loops: exp without max subtraction, on tiny inputs.
    for causal, (B, Hq, Hkv, nq, nk, d) in ((False, (2, 4, 2, 5, 7, 3)), (True, (1, 2, 1, 6, 8, 4)),
                                             (True, (1, 2, 2, 8, 3, 2)), (False, (1, 1, 1, 1, 1, 1))):
        q, k, v = _rand((B, Hq, nq, d), 8), _rand((B, Hkv, nk, d), 9), _rand((B, Hkv, nk, d), 10)
        scale = 0.6
        o, lse = fwd(q, k, v, scale, causal)
        g = Hq // Hkv
        for b in range(B):
            for h in range(Hq):
                for i in range(nq):
                    num = [0.0] * d
                    den = 0.0
                    for j in range(nk):
                        if causal and j > i + nk - nq:
                            continue
                        s = scale * sum(q[b, h, i, c] * k[b, h // g, j, c] for c in range(d))
                        w = math.exp(s)
                        den += w
                        for c in range(d):
                            num[c] += w * v[b, h // g, j, c]
                    if den == 0.0:
                        assert lse[b, h, i] == -math.inf and np.all(o[b, h, i] == 0.0)
                        continue
                    assert abs(lse[b, h, i] - math.log(den)) <= 1e-12
                    for c in range(d):
                        assert abs(o[b, h, i, c] - num[c] / den) <= 1e-12


def pin_library_sdpa(fwd):
    # torch's scaled_dot_product_attention in float64 on the CPU; with Nq = Nk
    # its causal flag equals the bottom-right mask.
    for causal in (False, True):
        q, k, v = _rand((2, 3, 33, 16), 11), _rand((2, 3, 33, 16), 12), _rand((2, 3, 33, 16), 13)
        o, _ = fwd(q, k, v, 0.3, causal)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), is_causal=causal, scale=0.3)
        np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)


def _online_two_tiles(q, k, v, scale, causal, tile):
    """Online softmax over K/V tiles (m, l, O with exp(old_m - new_m) rescale)."""
    nq, nk = q.shape[0], k.shape[0]
    o = np.zeros((nq, v.shape[1]))
    m = np.full(nq, -np.inf)
    l = np.zeros(nq)
    for j0 in range(0, nk, tile):
        j1 = min(nk, j0 + tile)
        s = scale * (q @ k[j0:j1].T)
        if causal:
            keys = np.arange(j0, j1)
            s = np.where(keys[None, :] <= np.arange(nq)[:, None] + nk - nq, s, -np.inf)
        m_new = np.maximum(m, s.max(axis=1))
        base = np.where(np.isfinite(m_new), m_new, 0.0)
        alpha = np.exp(np.where(np.isfinite(m), m - base, -np.inf))
        p = np.exp(s - base[:, None])
        l = alpha * l + p.sum(axis=1)
        o = alpha[:, None] * o + p @ v[j0:j1]
        m = m_new
    has = l > 0
    out = np.where(has[:, None], o / np.where(has, l, 1.0)[:, None], 0.0)
    lse = np.where(has, m + np.log(np.where(has, l, 1.0)), -np.inf)
    return out, lse


def pin_online_recurrence(fwd):
    for causal, nq, nk in ((False, 16, 16), (True, 16, 16), (True, 10, 16)):
        q, k, v = _rand((1, 1, nq, 8), 14), _rand((1, 1, nk, 8), 15) * 3, _rand((1, 1, nk, 8), 16)
        o, lse = fwd(q, k, v, 0.35, causal)
        o2, l2 = _online_two_tiles(q[0, 0], k[0, 0], v[0, 0], 0.35, causal, tile=nk // 2)
        np.testing.assert_allclose(o[0, 0], o2, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[0, 0], l2, rtol=0, atol=1e-12)


def pin_shift_invariance(fwd_shift):
    for causal in (False, True):
        q, k, v = _rand((1, 2, 9, 4), 17), _rand((1, 2, 9, 4), 18), _rand((1, 2, 9, 4), 19)
        r = _rand((1, 2, 9), 20) * 5
        o0, l0 = fwd_shift(q, k, v, 0.8, causal, None)
        o1, l1 = fwd_shift(q, k, v, 0.8, causal, r)
        np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l1, l0 + r, rtol=0, atol=1e-12)


def pin_permutation(fwd):
    q, k, v = _rand((1, 2, 6, 4), 21), _rand((1, 2, 10, 4), 22), _rand((1, 2, 10, 4), 23)
    perm = np.random.default_rng(24).permutation(10)
    o0, l0 = fwd(q, k, v, 0.5, False)
    o1, l1 = fwd(q, k[:, :, perm], v[:, :, perm], 0.5, False)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-12)


def pin_gqa_equals_repeated_heads(fwd):
    q, k, v = _rand((2, 8, 7, 4), 25), _rand((2, 2, 9, 4), 26), _rand((2, 2, 9, 4), 27)
    for causal in (False, True):
        o0, l0 = fwd(q, k, v, 0.5, causal)
        o1, l1 = fwd(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1), 0.5, causal)
        np.testing.assert_allclose(o0, o1, rtol=0, atol=1e-13)
        np.testing.assert_allclose(l0, l1, rtol=0, atol=1e-13)


def pin_varlen_equals_per_sequence(fwd_varlen):
    lens = [3, 1, 0, 7, 5]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q, k, v = _rand((4, T, 4), 28), _rand((2, T, 4), 29), _rand((2, T, 4), 30)
    for causal in (False, True):
        o, lse = fwd_varlen(q, k, v, 0.5, causal, cu)
        for s in range(len(lens)):
            t0, t1 = cu[s], cu[s + 1]
            if t1 == t0:
                continue
            os_, ls_ = attention_fwd(q[None, :, t0:t1], k[None, :, t0:t1], v[None, :, t0:t1], 0.5, causal)
            np.testing.assert_allclose(o[:, t0:t1], os_[0], rtol=0, atol=1e-13)
            np.testing.assert_allclose(lse[:, t0:t1], ls_[0], rtol=0, atol=1e-13)
        # Closed form independent of the per-sequence call: with Q = 0 each
        # row averages V over its own sequence's valid prefix.
        o0, l0 = fwd_varlen(np.zeros_like(q), k, v, 0.5, causal, cu)
        for s in range(len(lens)):
            t0, L = int(cu[s]), lens[s]
            for i in range(L):
                n = i + 1 if causal else L
                np.testing.assert_allclose(o0[:, t0 + i], v[:, t0:t0 + n].mean(axis=1).repeat(2, axis=0),
                                           rtol=0, atol=1e-13)
                np.testing.assert_allclose(l0[:, t0 + i], math.log(n), rtol=0, atol=1e-13)


def _pins():
    def fwd(q, k, v, scale, causal):
        return attention_fwd(q, k, v, scale, causal)

    def fwd_p(q, k, v, scale, causal):
        return attention_fwd(q, k, v, scale, causal, return_p=True)

    def fwd_shift(q, k, v, scale, causal, r):
        return attention_fwd(q, k, v, scale, causal, row_shift=r)

    def fwd_varlen(q, k, v, scale, causal, cu):
        return attention_fwd(q, k, v, scale, causal, cu_seqlens=cu)

    return [
        ("golden", lambda: pin_golden(fwd)),
        ("p_rows", lambda: pin_p_rows_sum_to_one(fwd_p)),
        ("zero_q", lambda: pin_zero_q_mean_of_v(fwd)),
        ("const_v", lambda: pin_constant_v(fwd)),
        ("brute", lambda: pin_brute_force(fwd)),
        ("sdpa", lambda: pin_library_sdpa(fwd)),
        ("online", lambda: pin_online_recurrence(fwd)),
        ("shift", lambda: pin_shift_invariance(fwd_shift)),
        ("perm", lambda: pin_permutation(fwd)),
        ("gqa", lambda: pin_gqa_equals_repeated_heads(fwd)),
        ("varlen", lambda: pin_varlen_equals_per_sequence(fwd_varlen)),
    ]


@pytest.mark.parametrize("name,check", _pins(), ids=[n for n, _ in _pins()])
def test_oracle_pin(name, check):
    check()


def test_golden_online_intermediates():
    """The hand-derived m, l and unnormalised O after each tile of row 0."""
    g, q, k, v = _golden_case()
    q, k, v = q[0, 0], k[0, 0], v[0, 0]
    m, l, o = -np.inf, 0.0, np.zeros(2)
    for t, (j0, j1) in enumerate(([0, 2], [2, 4])):
        s = q[0] @ k[j0:j1].T
        m_new = max(m, s.max())
        alpha = math.exp(m - m_new) if np.isfinite(m) else 0.0
        p = np.exp(s - m_new)
        l = alpha * l + p.sum()
        o = alpha * o + p @ v[j0:j1]
        m = m_new
        want = g["noncausal"]["online_row0"]["after_tile%d" % t]
        assert abs(m - math.log(want["m_exp"])) < 1e-15
        assert abs(l - float(Fraction(*want["l"]))) < 1e-15
        np.testing.assert_allclose(o, [float(Fraction(*x)) for x in want["O_unnormalised"]], atol=1e-15)


def test_fully_masked_rows():
    # Nq > Nk with the bottom-right causal mask: the first Nq - Nk rows see no key.
    q, k, v = _rand((1, 1, 6, 2), 31), _rand((1, 1, 2, 2), 32), _rand((1, 1, 2, 2), 33)
    o, lse = attention_fwd(q, k, v, 1.0, True)
    assert np.all(o[0, 0, :4] == 0.0) and np.all(lse[0, 0, :4] == -np.inf)
    assert np.all(np.isfinite(lse[0, 0, 4:]))
    o, lse = attention_fwd(q, k[:, :, :0], v[:, :, :0], 1.0, False)
    assert np.all(o == 0.0) and np.all(lse == -np.inf)


def test_rows_match_full():
    p = make_dense(1, 4, 2, 200, 300, 64, seed=7, causal=True)
    q, k, v = (bf16_bits_to_f64(x) for x in (p.q, p.k, p.v))
    o, lse = attention_fwd(q, k, v, p.scale, True)
    samples = [(0, 0, 0), (0, 3, 199), (0, 1, 57), (0, 2, 128)]
    o2, l2 = attention_rows(q, k, v, p.scale, True, samples)
    for n, (b, h, i) in enumerate(samples):
        np.testing.assert_array_equal(o2[n], o[b, h, i])
        assert l2[n] == lse[b, h, i]
    pv = make_varlen([5, 130, 1], 2, 1, 64, seed=8, causal=True)
    q, k, v = (bf16_bits_to_f64(x) for x in (pv.q, pv.k, pv.v))
    o, lse = attention_fwd(q, k, v, pv.scale, True, cu_seqlens=pv.cu_seqlens)
    samples = [(0, 1, 4), (1, 0, 129), (2, 1, 0), (1, 1, 0)]
    o2, l2 = attention_rows(q, k, v, pv.scale, True, samples, cu_seqlens=pv.cu_seqlens)
    for n, (s, h, i) in enumerate(samples):
        t = int(pv.cu_seqlens[s]) + i
        np.testing.assert_array_equal(o2[n], o[h, t])
        assert l2[n] == lse[h, t]


# --------------------------------------------------------------------------
# Planted mistakes: each broken copy of the per-head routine must fail a pin.
# --------------------------------------------------------------------------

def _mutant(kind):
    orig = oa._head_rows

    def head_rows(qh, kh, vh, rows, nq, scale, causal, row_shift, want_p):
        if kind == "no_scale":
            return orig(qh, kh, vh, rows, nq, 1.0, causal, row_shift, want_p)
        if kind == "k_for_v":
            return orig(qh, kh, kh, rows, nq, scale, causal, row_shift, want_p)
        if kind == "top_left_causal":
            return orig(qh, kh, vh, rows + (kh.shape[0] - nq), nq, scale, causal, row_shift, want_p)
        if kind == "causal_off_by_one":
            return orig(qh, kh, vh, rows - 1, nq, scale, causal, row_shift, want_p)
        if kind == "lse_without_max":
            o, lse, p = orig(qh, kh, vh, rows, nq, scale, causal, row_shift, want_p)
            s = scale * (qh @ kh.T)
            return o, lse - s.max(dim=1).values, p
        if kind == "exp2":
            # 2**s in place of e**s is e**(s ln 2): the scale silently shrinks.
            return orig(qh, kh, vh, rows, nq, scale * math.log(2.0), causal, row_shift, want_p)
        if kind == "unnormalised":
            o, lse, p = orig(qh, kh, vh, rows, nq, scale, causal, row_shift, want_p)
            return o * torch.exp(lse - lse.max())[:, None], lse, p
        if kind == "drop_last_key":
            o, lse, p = orig(qh, kh[:-1], vh[:-1], rows, nq, scale, causal, row_shift, want_p) \
                if kh.shape[0] > 1 else orig(qh, kh, vh, rows, nq, scale, causal, row_shift, want_p)
            return o, lse, (None if p is None else torch.cat([p, torch.zeros_like(p[:, :1])], dim=1))
        if kind == "q_transposed_heads":
            return orig(qh.flip(0), kh, vh, rows, nq, scale, causal, row_shift, want_p)
        raise AssertionError(kind)
    return head_rows


MUTANTS = ["no_scale", "k_for_v", "top_left_causal", "causal_off_by_one", "lse_without_max",
           "exp2", "unnormalised", "drop_last_key", "q_transposed_heads"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_planted_mistakes_are_caught(kind, monkeypatch):
    monkeypatch.setattr(oa, "_head_rows", _mutant(kind))
    failures = 0
    for _, check in _pins():
        try:
            check()
        except (AssertionError, ValueError, IndexError, RuntimeError):
            failures += 1
    assert failures > 0, "planted mistake %s passed every pin" % kind


@pytest.mark.parametrize("wrong", ["interleaved", "first_head"])
def test_gqa_mapping_mistake_is_caught(wrong, monkeypatch):
    """Query head h must read key/value head h // (Hq // Hkv)."""
    if wrong == "interleaved":
        monkeypatch.setattr(oa, "_kv_head", lambda h, g, hkv: h % hkv)
    else:
        monkeypatch.setattr(oa, "_kv_head", lambda h, g, hkv: 0)
    failures = 0
    for _, check in _pins():
        try:
            check()
        except (AssertionError, ValueError, IndexError, RuntimeError):
            failures += 1
    assert failures > 0
