"""Pins for the fp64 backward oracle (CPU only).

The oracle writes out the chain rule of O = softmax(scale Q K^T) V.  These
checks tie it to things other than its own formulas:
  * central finite differences of L = sum(O * dO) through the forward oracle;
  * float64 autograd through torch.softmax on the plain definition;
  * closed forms (a single key) and invariants that follow from the softmax
    being unchanged when a constant is added to every score of a row;
  * planted mistakes in the per-head routine, each of which must fail a pin.
"""
import math

import numpy as np
import pytest
import torch

import oracle.backward as ob
from oracle import attention_bwd, attention_bwd_keys, attention_bwd_rows, attention_fwd
from fa_inputs import bf16_bits_to_f64, make_dense


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _loss(q, k, v, do, scale, causal):
    o, _ = attention_fwd(q, k, v, scale, causal)
    return float((o * do).sum())


def _finite_diff(q, k, v, do, scale, causal, h=1e-5):
    grads = []
    for which in range(3):
        args = [q.copy(), k.copy(), v.copy()]
        x = args[which]
        g = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            x0 = x[idx]
            x[idx] = x0 + h
            lp = _loss(*args, do, scale, causal)
            x[idx] = x0 - h
            lm = _loss(*args, do, scale, causal)
            x[idx] = x0
            g[idx] = (lp - lm) / (2 * h)
        grads.append(g)
    return grads


# (B, Hq, Hkv, Nq, Nk, d, causal): GQA, Nq != Nk both ways, rows with no key.
FD_CASES = [(1, 2, 1, 3, 4, 3, False), (1, 2, 2, 4, 3, 2, True), (2, 2, 1, 3, 5, 2, True)]


def pin_finite_differences():
    for n, (B, Hq, Hkv, Nq, Nk, d, causal) in enumerate(FD_CASES):
        q, k, v = _rand((B, Hq, Nq, d), 10 + n), _rand((B, Hkv, Nk, d), 20 + n), _rand((B, Hkv, Nk, d), 30 + n)
        do = _rand((B, Hq, Nq, d), 40 + n)
        scale = 0.7
        dq, dk, dv, _ = attention_bwd(q, k, v, do, scale, causal)
        fq, fk, fv = _finite_diff(q, k, v, do, scale, causal)
        np.testing.assert_allclose(dq, fq, atol=1e-7, rtol=1e-6)
        np.testing.assert_allclose(dk, fk, atol=1e-7, rtol=1e-6)
        np.testing.assert_allclose(dv, fv, atol=1e-7, rtol=1e-6)


def pin_autograd():
    # Every row sees at least one key, so the masked softmax is defined.
    for n, (B, Hq, Hkv, Nq, Nk, d, causal) in enumerate([(1, 4, 2, 7, 9, 5, True), (2, 2, 2, 6, 6, 4, False)]):
        q, k, v = _rand((B, Hq, Nq, d), 50 + n), _rand((B, Hkv, Nk, d), 60 + n), _rand((B, Hkv, Nk, d), 70 + n)
        do = _rand((B, Hq, Nq, d), 80 + n)
        scale = 1.0 / math.sqrt(d)
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        g = Hq // Hkv
        kk = tk.repeat_interleave(g, dim=1)
        vv = tv.repeat_interleave(g, dim=1)
        s = scale * tq @ kk.transpose(-1, -2)
        if causal:
            i = torch.arange(Nq)[:, None]
            j = torch.arange(Nk)[None, :]
            s = s.masked_fill(j > i + (Nk - Nq), float("-inf"))
        o = torch.softmax(s, dim=-1) @ vv
        (o * torch.tensor(do)).sum().backward()
        dq, dk, dv, delta = attention_bwd(q, k, v, do, scale, causal)
        np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12, rtol=1e-10)
        np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12, rtol=1e-10)
        np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12, rtol=1e-10)
        np.testing.assert_allclose(delta, (o.detach().numpy() * do).sum(-1), atol=1e-12, rtol=1e-10)


def pin_single_key():
    """One key: P = 1 for every row, so O = V_0, dQ = dK = 0 and dV_0 = sum of dO."""
    B, Hq, Hkv, Nq, d = 1, 4, 2, 5, 3
    q, k, v = _rand((B, Hq, Nq, d), 1), _rand((B, Hkv, 1, d), 2), _rand((B, Hkv, 1, d), 3)
    do = _rand((B, Hq, Nq, d), 4)
    dq, dk, dv, delta = attention_bwd(q, k, v, do, 0.9, False)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13
    for kvh in range(Hkv):
        np.testing.assert_allclose(dv[0, kvh, 0], do[0, 2 * kvh:2 * kvh + 2].sum(axis=(0, 1)), atol=1e-13)
        for h in (2 * kvh, 2 * kvh + 1):
            np.testing.assert_allclose(delta[0, h], do[0, h] @ v[0, kvh, 0], atol=1e-13)


def pin_shift_invariants():
    """Adding c to every key leaves each row's softmax unchanged: sum_j dK_j = 0.
    sum_j P_ij = 1 on rows that see a key: sum_j dV_j = sum of those rows' dO.
    Q and K enter only through S: <dQ, Q> = <dK, K> for each key/value group."""
    B, Hq, Hkv, Nq, Nk, d = 2, 4, 2, 9, 6, 4
    q, k, v = _rand((B, Hq, Nq, d), 5), _rand((B, Hkv, Nk, d), 6), _rand((B, Hkv, Nk, d), 7)
    do = _rand((B, Hq, Nq, d), 8)
    g = Hq // Hkv
    for causal in (False, True):
        dq, dk, dv, _ = attention_bwd(q, k, v, do, 0.6, causal)
        np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
        seen = np.arange(Nq) + (Nk - Nq) >= 0 if causal else np.ones(Nq, bool)
        for b in range(B):
            for kvh in range(Hkv):
                hs = slice(kvh * g, (kvh + 1) * g)
                np.testing.assert_allclose(dv[b, kvh].sum(axis=0), do[b, hs][:, seen].sum(axis=(0, 1)),
                                           atol=1e-12)
                np.testing.assert_allclose((dq[b, hs] * q[b, hs]).sum(), (dk[b, kvh] * k[b, kvh]).sum(),
                                           atol=1e-11)


def pin_sampled_helpers():
    p = make_dense(1, 4, 2, 150, 170, 64, seed=9, causal=True)
    q, k, v = (bf16_bits_to_f64(x) for x in (p.q, p.k, p.v))
    do = _rand(q.shape, 12)
    dq, dk, dv, delta = attention_bwd(q, k, v, do, p.scale, True)
    rows = [0, 20, 149]
    gq, gd = attention_bwd_rows(q, k, v, do, p.scale, True, 0, 3, rows)
    np.testing.assert_allclose(gq, dq[0, 3, rows], atol=1e-12)
    np.testing.assert_allclose(gd, delta[0, 3, rows], atol=1e-12)
    keys = [0, 19, 169]
    gk, gv = attention_bwd_keys(q, k, v, do, p.scale, True, 0, 1, keys)
    np.testing.assert_allclose(gk, dk[0, 1, keys], atol=1e-12)
    np.testing.assert_allclose(gv, dv[0, 1, keys], atol=1e-12)


def pin_varlen_finite_differences():
    """Packed sequences: finite differences of sum(O * dO) through the forward
    oracle's own packed mode (sequences must not see each other)."""
    lens = [3, 1, 4]
    cu = np.array([0, 3, 4, 8], dtype=np.int32)
    Hq, Hkv, d, T = 2, 1, 2, 8
    q, k, v = _rand((Hq, T, d), 90), _rand((Hkv, T, d), 91), _rand((Hkv, T, d), 92)
    do = _rand((Hq, T, d), 93)
    scale = 0.8
    for causal in (False, True):
        dq, dk, dv, _ = attention_bwd(q, k, v, do, scale, causal, cu_seqlens=cu)

        def loss(qq, kk, vv):
            o, _ = attention_fwd(qq, kk, vv, scale, causal, cu_seqlens=cu)
            return float((o * do).sum())
        for grad, which in ((dq, 0), (dk, 1), (dv, 2)):
            args = [q.copy(), k.copy(), v.copy()]
            x = args[which]
            fd = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                x0 = x[idx]
                x[idx] = x0 + 1e-5
                lp = loss(*args)
                x[idx] = x0 - 1e-5
                lm = loss(*args)
                x[idx] = x0
                fd[idx] = (lp - lm) / 2e-5
            np.testing.assert_allclose(grad, fd, atol=1e-7, rtol=1e-6)
    assert lens == [int(cu[i + 1] - cu[i]) for i in range(3)]


PINS = [("finite_differences", pin_finite_differences), ("varlen_finite_differences", pin_varlen_finite_differences),
        ("autograd", pin_autograd),
        ("single_key", pin_single_key), ("shift_invariants", pin_shift_invariants),
        ("sampled_helpers", pin_sampled_helpers)]


@pytest.mark.parametrize("name,check", PINS, ids=[n for n, _ in PINS])
def test_oracle_bwd_pin(name, check):
    check()


# --------------------------------------------------------------------------
# Planted mistakes in the per-head backward: each must fail at least one pin.
# --------------------------------------------------------------------------

def _mutant(kind):
    def head_grads(qh, kh, vh, dob, rows, nq, scale, causal):
        o, _, p = ob._head_rows(qh, kh, vh, rows, nq, scale, causal, None, True)
        dv = p.T @ dob
        dp = dob @ vh.T
        dlt = (dob * o).sum(dim=1)
        if kind == "no_delta":
            ds = p * dp
        elif kind == "delta_sign":
            ds = p * (dp + dlt[:, None])
        elif kind == "delta_from_q":
            ds = p * (dp - (qh * o).sum(dim=1)[:, None])
        else:
            ds = p * (dp - dlt[:, None])
        dq = scale * (ds @ kh)
        dk = scale * (ds.T @ qh)
        if kind == "dq_no_scale":
            dq = ds @ kh
        if kind == "dk_from_do":
            dk = scale * (ds.T @ dob)
        if kind == "dv_from_dp":
            dv = (p * dp).T @ dob
        if kind == "dv_unmasked":
            dv = torch.softmax(scale * (qh @ kh.T), dim=1).T @ dob
        if kind == "dq_uses_v":
            dq = scale * (ds @ vh)
        return dq, dk, dv, dlt
    return head_grads


BWD_MUTANTS = ["no_delta", "delta_sign", "delta_from_q", "dq_no_scale", "dk_from_do", "dv_from_dp",
               "dv_unmasked", "dq_uses_v"]


@pytest.mark.parametrize("kind", BWD_MUTANTS)
def test_planted_bwd_mistakes_are_caught(kind, monkeypatch):
    monkeypatch.setattr(ob, "_head_grads", _mutant(kind))
    failures = 0
    for _, check in PINS:
        try:
            check()
        except (AssertionError, ValueError, IndexError, RuntimeError):
            failures += 1
    assert failures > 0, "planted mistake %s passed every pin" % kind


def test_gqa_sum_mistake_is_caught(monkeypatch):
    """dK and dV of a key/value head sum over its query heads."""
    monkeypatch.setattr(ob, "_kv_head", lambda h, g, hkv: h % hkv)
    failures = 0
    for _, check in PINS:
        try:
            check()
        except (AssertionError, ValueError, IndexError, RuntimeError):
            failures += 1
    assert failures > 0
