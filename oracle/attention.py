"""fp64 CPU oracle for the exact attention forward pass.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module;
only the tests, the smoke check and the bench's CPU-baseline leg may call it.

It is the plain definition of standard attention, written out in float64 with
the full score row materialised and a two-pass softmax (no online recurrence):

    S = scale * Q K^T,  P = softmax(S) row-wise,  O = P V

("FlashAttention面试讲解" interview canvas, element ``std-text``: standard
attention forms the N x N score matrix, applies softmax, then multiplies by V).
The same canvas (elements ``flash-text`` and ``v1-card-body``) states that the
tiled method is not an approximation and does not change the mathematical
result, so the plain definition is the exact target of the tiled kernel.

Readings taken where the pages are silent (each one is listed with its
justification in the design notes):

* per-row statistic: the forward pass keeps "the output and a few per-row
  statistics" (``v1-card-body``, ``qa3-a``); the single statistic emitted is
  LSE_i = ln sum_j exp(S_ij) over the valid keys (natural log, scaled scores).
* causal mask: bottom-right aligned, key j is valid for query i when
  j <= i + (Nk - Nq).
* a row with no valid key gets O = 0 and LSE = -inf.
* grouped-query attention: query head h reads key/value head h // (Hq // Hkv).
* packed variable-length batches: one ``cu_seqlens`` array shared by queries
  and keys; each sequence attends only within itself.

Query rows are independent under the definition, so rows are processed in
groups to bound memory; nothing inside a row is reordered or fused.

Pins: the oracle is checked against closed forms, invariants, brute force on
tiny inputs, a library routine and hand-derived golden values in
``tests/test_oracle.py``.
"""
from __future__ import annotations

from typing import Iterable, Optional, Sequence, Tuple

import numpy as np
import torch

_ROW_BLOCK = 512


def _as_f64(x) -> torch.Tensor:
    return torch.as_tensor(np.asarray(x, dtype=np.float64))


def _head_rows(qh: torch.Tensor, kh: torch.Tensor, vh: torch.Tensor, rows: torch.Tensor,
               nq: int, scale: float, causal: bool, row_shift: Optional[torch.Tensor],
               want_p: bool):
    """Attention for the query rows ``rows`` of one head (all float64).

    qh: [len(rows), d] query vectors of those rows, kh/vh: [Nk, d].
    Returns O [len(rows), d], LSE [len(rows)] and optionally P.
    """
    nk = kh.shape[0]
    # S = scale * q . k for every key (the full score row, materialised).
    s = scale * (qh @ kh.T)
    if row_shift is not None:
        s = s + row_shift[:, None]
    keys = torch.arange(nk, dtype=torch.int64)
    if causal:
        valid = keys[None, :] <= (rows[:, None] + (nk - nq))
    else:
        valid = torch.ones((rows.numel(), nk), dtype=torch.bool)
    neg_inf = torch.tensor(float("-inf"), dtype=torch.float64)
    s_valid = torch.where(valid, s, neg_inf)
    # Pass 1: row maximum over the valid keys.
    m = s_valid.max(dim=1).values if nk > 0 else torch.full((rows.numel(),), float("-inf"),
                                                             dtype=torch.float64)
    has_key = valid.any(dim=1) if nk > 0 else torch.zeros(rows.numel(), dtype=torch.bool)
    m_safe = torch.where(has_key, m, torch.zeros_like(m))
    # Pass 2: exponentials, their sum, normalised probabilities.
    e = torch.where(valid, torch.exp(s - m_safe[:, None]), torch.zeros_like(s))
    denom = e.sum(dim=1)
    p = torch.where(has_key[:, None], e / torch.where(has_key, denom, torch.ones_like(denom))[:, None],
                    torch.zeros_like(e))
    o = p @ vh
    lse = torch.where(has_key, m_safe + torch.log(torch.where(has_key, denom, torch.ones_like(denom))),
                      neg_inf.expand_as(m))
    return o, lse, (p if want_p else None)


def _kv_head(h: int, g: int, hkv: int) -> int:
    """Key/value head read by query head h: contiguous groups of g query heads."""
    return h // g


def _check_shapes(q, k, v, cu_seqlens):
    if cu_seqlens is None:
        assert q.ndim == 4 and k.ndim == 4 and v.ndim == 4
        B, Hq, Nq, d = q.shape
        assert k.shape[0] == B and k.shape == v.shape and k.shape[3] == d
        Hkv = k.shape[1]
    else:
        assert q.ndim == 3 and k.ndim == 3 and v.ndim == 3
        Hq, T, d = q.shape
        assert k.shape == v.shape and k.shape[1] == T and k.shape[2] == d
        Hkv = k.shape[0]
    assert Hkv >= 1 and Hq % Hkv == 0, "Hq must be a multiple of Hkv"
    return Hq // Hkv


def attention_fwd(q, k, v, scale: float, causal: bool, cu_seqlens=None,
                  row_shift=None, return_p: bool = False):
    """Exact attention forward in float64.

    Dense: q [B, Hq, Nq, d], k/v [B, Hkv, Nk, d]; returns O [B, Hq, Nq, d]
    and LSE [B, Hq, Nq].  Packed: q [Hq, T, d], k/v [Hkv, T, d] with
    ``cu_seqlens`` [nseq+1]; returns O [Hq, T, d] and LSE [Hq, T].

    ``row_shift`` (same leading shape as LSE) is added to row i of S before the
    softmax; it exists only so a test can check shift invariance.
    ``return_p`` also returns the probability matrices (dense only; keep the
    shapes tiny).
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    g = _check_shapes(q, k, v, cu_seqlens)
    shift = None if row_shift is None else _as_f64(row_shift)
    if cu_seqlens is None:
        B, Hq, Nq, d = q.shape
        Nk = k.shape[2]
        o = torch.zeros((B, Hq, Nq, d), dtype=torch.float64)
        lse = torch.zeros((B, Hq, Nq), dtype=torch.float64)
        ps = torch.zeros((B, Hq, Nq, Nk), dtype=torch.float64) if return_p else None
        for b in range(B):
            for h in range(Hq):
                kvh = _kv_head(h, g, k.shape[-3])
                for r0 in range(0, Nq, _ROW_BLOCK):
                    r1 = min(Nq, r0 + _ROW_BLOCK)
                    rows = torch.arange(r0, r1, dtype=torch.int64)
                    sh = None if shift is None else shift[b, h, r0:r1]
                    ob, lb, pb = _head_rows(q[b, h, r0:r1], k[b, kvh], v[b, kvh], rows, Nq,
                                            scale, causal, sh, return_p)
                    o[b, h, r0:r1] = ob
                    lse[b, h, r0:r1] = lb
                    if return_p:
                        ps[b, h, r0:r1] = pb
        out = (o.numpy(), lse.numpy())
        return out + (ps.numpy(),) if return_p else out
    assert not return_p, "return_p is for dense tiny shapes"
    cu = [int(x) for x in np.asarray(cu_seqlens)]
    Hq, T, d = q.shape
    o = torch.zeros((Hq, T, d), dtype=torch.float64)
    lse = torch.zeros((Hq, T), dtype=torch.float64)
    for s in range(len(cu) - 1):
        t0, t1 = cu[s], cu[s + 1]
        L = t1 - t0
        for h in range(Hq):
            kvh = _kv_head(h, g, k.shape[-3])
            for r0 in range(0, L, _ROW_BLOCK):
                r1 = min(L, r0 + _ROW_BLOCK)
                rows = torch.arange(r0, r1, dtype=torch.int64)
                sh = None if shift is None else shift[h, t0 + r0:t0 + r1]
                ob, lb, _ = _head_rows(q[h, t0 + r0:t0 + r1], k[kvh, t0:t1], v[kvh, t0:t1], rows, L,
                                       scale, causal, sh, False)
                o[h, t0 + r0:t0 + r1] = ob
                lse[h, t0 + r0:t0 + r1] = lb
    return o.numpy(), lse.numpy()


def attention_rows(q, k, v, scale: float, causal: bool, samples: Sequence[Tuple[int, int, int]],
                   cu_seqlens=None):
    """The same definition for a sample of single output rows.

    Dense: each sample is (b, h, i).  Packed: each sample is (seq, h, i) with i
    local to the sequence.  Returns O [n, d] and LSE [n] in sample order.
    Arrays may be float64 or anything numpy widens to float64 exactly.
    """
    g = _check_shapes(q, k, v, cu_seqlens)
    d = q.shape[-1]
    o = np.zeros((len(samples), d), dtype=np.float64)
    lse = np.zeros(len(samples), dtype=np.float64)
    cu = None if cu_seqlens is None else [int(x) for x in np.asarray(cu_seqlens)]
    for n, (b, h, i) in enumerate(samples):
        kvh = _kv_head(h, g, k.shape[-3])
        if cu is None:
            nq = q.shape[2]
            qi = _as_f64(q[b, h, i:i + 1])
            kh, vh = _as_f64(k[b, kvh]), _as_f64(v[b, kvh])
        else:
            t0, t1 = cu[b], cu[b + 1]
            nq = t1 - t0
            qi = _as_f64(q[h, t0 + i:t0 + i + 1])
            kh, vh = _as_f64(k[kvh, t0:t1]), _as_f64(v[kvh, t0:t1])
        ob, lb, _ = _head_rows(qi, kh, vh, torch.tensor([i], dtype=torch.int64), nq,
                               scale, causal, None, False)
        o[n] = ob[0].numpy()
        lse[n] = float(lb[0])
    return o, lse


def oracle_threads() -> int:
    """Host threads the oracle's tensor operations run on."""
    return torch.get_num_threads()
