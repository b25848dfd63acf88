"""fp64 CPU oracle for the exact attention backward pass.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module;
only the tests and the bench's CPU-baseline leg may call it.

The pages say what the backward pass keeps and recomputes, not its formulas.
The forward pass stores only the output and per-row statistics, and the
backward pass recomputes the local scores and probabilities instead of
reading a stored N x N matrix ("FlashAttention面试讲解" interview canvas,
elements ``v1-card-body`` and ``qa3-a``).  What the backward pass computes is
therefore fixed by the forward definition alone: the gradients of

    O = softmax(scale * Q K^T) V      (element ``std-text``)

with respect to Q, K and V, for an upstream gradient dO.  Written out by the
chain rule, per head:

    P  = softmax(S),  S = scale * Q K^T        (masked entries: P = 0)
    dV = P^T dO
    dP = dO V^T
    D_i = sum_j P_ij dP_ij  ( = dO_i . O_i )
    dS = P * (dP - D)                            (softmax Jacobian, row-wise)
    dQ = scale * dS K
    dK = scale * dS^T Q

Under grouped-query attention a key/value head is read by ``Hq / Hkv`` query
heads, so its dK and dV are the sums over those heads.  Rows with no visible
key have P = 0 and contribute nothing.

P comes from the forward oracle's own materialised, two-pass softmax, and
every product is a float64 matmul.  Nothing is blocked, fused or reordered.

Pins (``tests/test_oracle_bwd.py``): central finite differences of
L = sum(O * dO) on tiny inputs, float64 autograd through torch.softmax,
closed forms (a single key), and invariants that follow from the softmax's
shift invariance.
"""
from __future__ import annotations

import numpy as np
import torch

from .attention import _as_f64, _check_shapes, _head_rows, _kv_head

_ROW_BLOCK = 512


def _head_grads(qh, kh, vh, dob, rows, nq: int, scale: float, causal: bool):
    """Backward of one head for the query rows ``rows`` (all float64).

    qh, dob: [len(rows), d] queries and output gradients of those rows;
    kh, vh: [Nk, d].  Returns dQ [len(rows), d], this block's contributions
    to dK and dV [Nk, d], and delta [len(rows)].
    """
    o, _, p = _head_rows(qh, kh, vh, rows, nq, scale, causal, None, True)
    dv = p.T @ dob                       # dV = P^T dO
    dp = dob @ vh.T                      # dP = dO V^T
    dlt = (dob * o).sum(dim=1)           # D_i = dO_i . O_i
    ds = p * (dp - dlt[:, None])         # dS = P * (dP - D)
    dq = scale * (ds @ kh)               # dQ = scale dS K
    dk = scale * (ds.T @ qh)             # dK = scale dS^T Q
    return dq, dk, dv, dlt


def attention_bwd(q, k, v, do, scale: float, causal: bool, cu_seqlens=None):
    """Gradients of exact attention in float64.

    Dense: q, do [B, Hq, Nq, d]; k, v [B, Hkv, Nk, d].  Returns numpy float64
    arrays dq [B, Hq, Nq, d], dk and dv [B, Hkv, Nk, d], and the per-row
    statistic delta [B, Hq, Nq] = rowsum(dO * O).
    Packed (``cu_seqlens`` [nseq+1]): q, do [Hq, T, d]; k, v [Hkv, T, d]; each
    sequence attends only within itself, so its gradients are those of the
    dense problem made of that sequence alone; returns dq [Hq, T, d], dk, dv
    [Hkv, T, d] and delta [Hq, T].
    """
    if cu_seqlens is not None:
        q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
        cu = [int(x) for x in np.asarray(cu_seqlens)]
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        delta = np.zeros(q.shape[:2])
        for s in range(len(cu) - 1):
            t0, t1 = cu[s], cu[s + 1]
            if t1 == t0:
                continue
            a, b_, c, d_ = attention_bwd(q[None, :, t0:t1], k[None, :, t0:t1], v[None, :, t0:t1],
                                         do[None, :, t0:t1], scale, causal)
            dq[:, t0:t1], dk[:, t0:t1], dv[:, t0:t1], delta[:, t0:t1] = a[0], b_[0], c[0], d_[0]
        return dq, dk, dv, delta
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    g = _check_shapes(q, k, v, None)
    assert do.shape == q.shape
    B, Hq, Nq, d = q.shape
    Hkv = k.shape[1]
    dq = torch.zeros_like(q)
    dk = torch.zeros_like(k)
    dv = torch.zeros_like(v)
    delta = torch.zeros((B, Hq, Nq), dtype=torch.float64)
    for b in range(B):
        for h in range(Hq):
            kvh = _kv_head(h, g, Hkv)
            for r0 in range(0, Nq, _ROW_BLOCK):
                r1 = min(Nq, r0 + _ROW_BLOCK)
                rows = torch.arange(r0, r1, dtype=torch.int64)
                gq, gk, gv, dlt = _head_grads(q[b, h, r0:r1], k[b, kvh], v[b, kvh], do[b, h, r0:r1], rows, Nq,
                                              scale, causal)
                dq[b, h, r0:r1] = gq
                dk[b, kvh] += gk
                dv[b, kvh] += gv
                delta[b, h, r0:r1] = dlt
    return dq.numpy(), dk.numpy(), dv.numpy(), delta.numpy()


def attention_bwd_rows(q, k, v, do, scale: float, causal: bool, b: int, h: int, rows):
    """dQ and delta of selected query rows of one head (float64).

    Rows are independent for dQ, so sampled rows of a large problem can be
    checked without the whole backward pass.  Returns (dq [len(rows), d],
    delta [len(rows)]).
    """
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    g = _check_shapes(q, k, v, None)
    Nq = q.shape[2]
    kvh = _kv_head(h, g, k.shape[1])
    rows_t = torch.as_tensor(np.asarray(rows, dtype=np.int64))
    gq, _, _, dlt = _head_grads(q[b, h][rows_t], k[b, kvh], v[b, kvh], do[b, h][rows_t], rows_t, Nq, scale,
                                causal)
    return gq.numpy(), dlt.numpy()


def attention_bwd_keys(q, k, v, do, scale: float, causal: bool, b: int, kvh: int, keys):
    """dK and dV of selected keys of one key/value head (float64).

    A key's gradient sums over every query row of the group's heads, so this
    runs the whole head group and keeps the requested keys.  Returns
    (dk [len(keys), d], dv [len(keys), d]).
    """
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    g = _check_shapes(q, k, v, None)
    Nq = q.shape[2]
    keys_t = torch.as_tensor(np.asarray(keys, dtype=np.int64))
    d = q.shape[3]
    dk = torch.zeros((keys_t.numel(), d), dtype=torch.float64)
    dv = torch.zeros((keys_t.numel(), d), dtype=torch.float64)
    for h in range(kvh * g, (kvh + 1) * g):
        for r0 in range(0, Nq, _ROW_BLOCK):
            r1 = min(Nq, r0 + _ROW_BLOCK)
            rows = torch.arange(r0, r1, dtype=torch.int64)
            _, gk, gv, _ = _head_grads(q[b, h, r0:r1], k[b, kvh], v[b, kvh], do[b, h, r0:r1], rows, Nq, scale,
                                       causal)
            dk += gk[keys_t]
            dv += gv[keys_t]
    return dk.numpy(), dv.numpy()
