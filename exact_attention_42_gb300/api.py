"""PyTorch-facing wrapper: checks tensors, allocates outputs, calls fa_fwd.

PyTorch supplies device memory and the current stream only; every step of
the attention computation runs in the library's CUDA kernel.
"""
from __future__ import annotations

import functools
import math
import os
from typing import Optional, Tuple

import torch

from ._lib import FaError, fa_bwd, fa_fp8_quantize, fa_fwd, fa_fwd_fp8, fa_fwd_host

# NVTX ranges around every entry point, for profilers that show them (ncu's
# --nvtx filters, for one): on when FA_NVTX is set to a non-zero value.
NVTX = os.environ.get("FA_NVTX", "") not in ("", "0")


def _nvtx(name: str):
    def wrap(fn):
        @functools.wraps(fn)
        def call(*args, **kwargs):
            if not NVTX:
                return fn(*args, **kwargs)
            torch.cuda.nvtx.range_push(name)
            try:
                return fn(*args, **kwargs)
            finally:
                torch.cuda.nvtx.range_pop()
        return call
    return wrap


def _check(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int, device) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if t.dim() != ndim:
        raise ValueError("%s must have %d dims, got shape %s" % (name, ndim, tuple(t.shape)))
    if not t.is_cuda or (device is not None and t.device != device):
        raise ValueError("%s must be on the same CUDA device as q" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


@_nvtx("fa.fwd")
def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
        scale: Optional[float] = None, cu_seqlens: Optional[torch.Tensor] = None,
        out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
        stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Exact attention forward on the GPU; returns (O, LSE).

    Dense: q [B, Hq, Nq, d], k/v [B, Hkv, Nk, d] -> O like q, LSE [B, Hq, Nq] fp32.
    Packed (cu_seqlens int32 [nseq+1] on the device): q [Hq, T, d], k/v [Hkv, T, d]
    -> O [Hq, T, d], LSE [Hq, T].  Inputs are bf16, contiguous, on one GPU; d is
    64 or 128; scale defaults to 1/sqrt(d).  Runs on ``stream`` (default: the
    current stream) without synchronising.
    """
    dev = q.device
    packed = cu_seqlens is not None
    nd = 3 if packed else 4
    _check(q, "q", torch.bfloat16, nd, None)
    _check(k, "k", torch.bfloat16, nd, dev)
    _check(v, "v", torch.bfloat16, nd, dev)
    if k.shape != v.shape:
        raise ValueError("k and v must have the same shape")
    if packed:
        _check(cu_seqlens, "cu_seqlens", torch.int32, 1, dev)
        Hq, T, d = q.shape
        Hkv, Tk, dk = k.shape
        if Tk != T or dk != d:
            raise ValueError("packed q, k, v must share the token count and head dim")
        B, Nq, Nk = cu_seqlens.numel() - 1, T, T
        o_shape, lse_shape = (Hq, T, d), (Hq, T)
    else:
        B, Hq, Nq, d = q.shape
        Bk, Hkv, Nk, dk = k.shape
        if Bk != B or dk != d:
            raise ValueError("q and k must share batch size and head dim")
        o_shape, lse_shape = (B, Hq, Nq, d), (B, Hq, Nq)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(o_shape, dtype=torch.bfloat16, device=dev)
    else:
        _check(out, "out", torch.bfloat16, nd, dev)
        if tuple(out.shape) != o_shape:
            raise ValueError("out has shape %s, expected %s" % (tuple(out.shape), o_shape))
    if lse is None:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    else:
        _check(lse, "lse", torch.float32, nd - 1, dev)
        if tuple(lse.shape) != lse_shape:
            raise ValueError("lse has shape %s, expected %s" % (tuple(lse.shape), lse_shape))
    with torch.cuda.device(dev):
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        st = fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                    B, Hq, Hkv, Nq, Nk, d, float(scale), int(bool(causal)),
                    cu_seqlens.data_ptr() if packed else None, s.cuda_stream)
    if st != 0:
        raise FaError(st)
    return out, lse


@_nvtx("fa.fwd_host")
def fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
             scale: Optional[float] = None, cu_seqlens: Optional[torch.Tensor] = None,
             device: Optional[torch.device] = None, out: Optional[torch.Tensor] = None,
             lse: Optional[torch.Tensor] = None, chunks: int = 4) -> Tuple[torch.Tensor, torch.Tensor]:
    """The forward for host tensors, through the C entry fa_fwd_host: copies
    the inputs to the GPU, runs the kernel, copies O and LSE back to host
    memory and waits for the result.

    Dense inputs are processed in about ``chunks`` pieces, each a contiguous
    (batch, key/value head range) slice with its query heads; the library
    overlaps one piece's copies with the kernel and the copies of others (on
    GB300 the host-to-device copies of the B2/H32/N4096 inputs then bound the
    call).  Inputs in pinned memory make the copies asynchronous; ``out`` /
    ``lse`` (host tensors of O's and LSE's shapes, pinned for overlap) receive
    the results, otherwise they are allocated, pinned when the inputs are.
    Packed batches (``cu_seqlens`` int32 on the host) take one piece.  The
    device staging buffers are allocated here, through PyTorch.
    """
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    packed = cu_seqlens is not None
    nd = 3 if packed else 4
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.dim() != nd or t.is_cuda \
                or not t.is_contiguous():
            raise ValueError("%s must be a contiguous bf16 host tensor with %d dims" % (name, nd))
    if k.shape != v.shape:
        raise ValueError("k and v must have the same shape")
    if packed:
        if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or cu_seqlens.is_cuda:
            raise ValueError("cu_seqlens must be an int32 host tensor")
        cu_seqlens = cu_seqlens.contiguous()
        Hq, Nq, d = q.shape
        Hkv, Nk, _ = k.shape
        B = cu_seqlens.numel() - 1
    else:
        B, Hq, Nq, d = q.shape
        _, Hkv, Nk, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None or lse is None:
        nb = q.is_pinned()  # a driver query: only when outputs are allocated here
        if out is None:
            out = torch.empty(q.shape, dtype=q.dtype, pin_memory=nb)
        if lse is None:
            lse = torch.empty(q.shape[:-1], dtype=torch.float32, pin_memory=nb)
    if tuple(out.shape) != tuple(q.shape) or out.dtype != torch.bfloat16 or out.is_cuda or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 host tensor shaped like q")
    if tuple(lse.shape) != tuple(q.shape[:-1]) or lse.dtype != torch.float32 or lse.is_cuda \
            or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 host tensor of q's leading shape")
    # One staging allocation for Q, K, V, O, LSE (and cu_seqlens), carved at
    # 256-byte offsets: the C entry needs 16-byte aligned Q, K, V, O and
    # 4-byte aligned LSE and cu_seqlens.  It lives until the call has waited.
    sizes = (q.numel() * 2, k.numel() * 2, v.numel() * 2, q.numel() * 2, out.numel() // d * 4,
             cu_seqlens.numel() * 4 if packed else 0)
    offs, total = [], 0
    for n in sizes:
        offs.append(total)
        total += (n + 255) // 256 * 256
    if device.index != torch.cuda.current_device():
        with torch.cuda.device(device):
            return _fwd_host_call(q, k, v, out, lse, cu_seqlens, sizes, offs, total, B, Hq, Hkv, Nq, Nk, d, scale,
                                  causal, chunks, device)
    return _fwd_host_call(q, k, v, out, lse, cu_seqlens, sizes, offs, total, B, Hq, Hkv, Nq, Nk, d, scale, causal,
                          chunks, device)


def _fwd_host_call(q, k, v, out, lse, cu_seqlens, sizes, offs, total, B, Hq, Hkv, Nq, Nk, d, scale, causal, chunks,
                   device):
    """fwd_host's C call on the current device, which is `device`."""
    stage = torch.empty(max(total, 1), dtype=torch.uint8, device=device)
    base = stage.data_ptr()
    qd, kd, vd, od, ld, cud = (base + off if n else 0 for n, off in zip(sizes, offs))
    packed = cu_seqlens is not None
    s = torch.cuda.current_stream(device)
    st = fa_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                     qd or None, kd or None, vd or None, od or None, ld or None,
                     B, Hq, Hkv, Nq, Nk, d, float(scale), int(bool(causal)),
                     cu_seqlens.data_ptr() if packed else None, cud if packed else None,
                     max(1, int(chunks)), s.cuda_stream)
    if st != 0:
        raise FaError(st, "fa_fwd_host")
    s.synchronize()
    return out, lse


@_nvtx("fa.bwd")
def bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
        dout: torch.Tensor, causal: bool = False, scale: Optional[float] = None,
        stream: Optional[torch.cuda.Stream] = None, dq: Optional[torch.Tensor] = None,
        dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None,
        delta: Optional[torch.Tensor] = None, cu_seqlens: Optional[torch.Tensor] = None):
    """Gradients of exact attention on the GPU; returns (dQ, dK, dV, delta).

    Dense: q, o, dout [B, Hq, Nq, d], k/v [B, Hkv, Nk, d] bf16, lse [B, Hq, Nq]
    fp32 from ``fwd`` on the same inputs; delta [B, Hq, Nq] fp32 is
    rowsum(dout * o).  Packed (cu_seqlens int32 [nseq+1] on the device): the
    [H, T, d] / [H, T] layouts of ``fwd``.  Output tensors may be passed in
    (dq, dk, dv, delta), otherwise they are allocated.  Runs on ``stream``
    (default: the current stream) without synchronising.
    """
    dev = q.device
    packed = cu_seqlens is not None
    nd = 3 if packed else 4
    _check(q, "q", torch.bfloat16, nd, None)
    for t, n in ((k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _check(t, n, torch.bfloat16, nd, dev)
    _check(lse, "lse", torch.float32, nd - 1, dev)
    if packed:
        _check(cu_seqlens, "cu_seqlens", torch.int32, 1, dev)
        Hq, Nq, d = q.shape
        Hkv, Nk, dk_ = k.shape
        B = cu_seqlens.numel() - 1
        if Nk != Nq or dk_ != d or tuple(v.shape) != tuple(k.shape):
            raise ValueError("packed k and v must be [Hkv, T, d] with q's T and d")
        row_shape = (Hq, Nq)
    else:
        B, Hq, Nq, d = q.shape
        Bk, Hkv, Nk, dk_ = k.shape
        if Bk != B or dk_ != d or tuple(v.shape) != tuple(k.shape):
            raise ValueError("k and v must be [B, Hkv, Nk, d] with q's B and d")
        row_shape = (B, Hq, Nq)
    if tuple(o.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape):
        raise ValueError("o and dout must have q's shape")
    if tuple(lse.shape) != row_shape:
        raise ValueError("lse must be %s" % (row_shape,))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    def out(t, like, name, dtype=torch.bfloat16):
        if t is None:
            return torch.empty(like, dtype=dtype, device=dev)
        _check(t, name, dtype, len(like), dev)
        if tuple(t.shape) != tuple(like):
            raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(like)))
        return t
    dq = out(dq, q.shape, "dq")
    dk = out(dk, k.shape, "dk")
    dv = out(dv, v.shape, "dv")
    delta = out(delta, row_shape, "delta", torch.float32)
    with torch.cuda.device(dev):
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        st = fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                    dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), delta.data_ptr(), B, Hq, Hkv, Nq, Nk, d,
                    float(scale), int(bool(causal)), cu_seqlens.data_ptr() if packed else None, s.cuda_stream)
    if st != 0:
        raise FaError(st, "fa_bwd")
    return dq, dk, dv, delta


@_nvtx("fa.fwd_fp8")
def fwd_fp8(q8: torch.Tensor, k8: torch.Tensor, vt8: torch.Tensor, q_descale: torch.Tensor,
            k_descale: torch.Tensor, v_descale: torch.Tensor, causal: bool = False, scale: Optional[float] = None,
            out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
            stream: Optional[torch.cuda.Stream] = None,
            cu_seqlens: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Attention forward with e4m3 inputs on the GPU; returns (O bf16, LSE fp32).

    Dense: q8 [B, Hq, Nq, d], k8 [B, Hkv, Nk, d] and vt8 [B, Hkv, d, Nk] hold
    e4m3 codes (torch.uint8 or torch.float8_e4m3fn), d = 64 or 128; the
    descales are fp32 [B, Hq], [B, Hkv], [B, Hkv].  Nk must be a multiple of 16.
    Packed (cu_seqlens int32 [nseq+1] on the device): q8 [Hq, T, d],
    k8 [Hkv, T, d], vt8 [Hkv, d, T] and descales [Hq], [Hkv], [Hkv] (one per
    head); T must be a multiple of 16.
    """
    dev = q8.device
    as_u8 = lambda t: t.view(torch.uint8) if t.dtype != torch.uint8 else t
    q8, k8, vt8 = as_u8(q8), as_u8(k8), as_u8(vt8)
    packed = cu_seqlens is not None
    nd = 3 if packed else 4
    _check(q8, "q8", torch.uint8, nd, None)
    _check(k8, "k8", torch.uint8, nd, dev)
    _check(vt8, "vt8", torch.uint8, nd, dev)
    if packed:
        _check(cu_seqlens, "cu_seqlens", torch.int32, 1, dev)
        Hq, Nq, d = q8.shape
        Hkv, Nk, dk = k8.shape
        B = cu_seqlens.numel() - 1
        if Nk != Nq or dk != d or tuple(vt8.shape) != (Hkv, d, Nk):
            raise ValueError("packed k8 must be [Hkv, T, d] and vt8 [Hkv, d, T] with q8's T and d")
        shapes = ((Hq,), (Hkv,), (Hkv,))
        row_shape = (Hq, Nq)
    else:
        B, Hq, Nq, d = q8.shape
        Bk, Hkv, Nk, dk = k8.shape
        if Bk != B or dk != d or tuple(vt8.shape) != (B, Hkv, d, Nk):
            raise ValueError("k8 must be [B, Hkv, Nk, d] and vt8 [B, Hkv, d, Nk]")
        shapes = ((B, Hq), (B, Hkv), (B, Hkv))
        row_shape = (B, Hq, Nq)
    for t, n, shp in zip((q_descale, k_descale, v_descale), ("q_descale", "k_descale", "v_descale"), shapes):
        _check(t, n, torch.float32, len(shp), dev)
        if tuple(t.shape) != shp:
            raise ValueError("%s must be %s" % (n, shp))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(tuple(q8.shape), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(row_shape, dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        st = fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), vt8.data_ptr(), q_descale.data_ptr(), k_descale.data_ptr(),
                        v_descale.data_ptr(), out.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Nq, Nk, d, float(scale),
                        int(bool(causal)), cu_seqlens.data_ptr() if packed else None, s.cuda_stream)
    if st != 0:
        raise FaError(st, "fa_fwd_fp8")
    return out, lse


def hadamard_signs(d: int, seed: int, device=None) -> torch.Tensor:
    """A seeded vector of d random signs (+1 / -1, int8) for ``fp8_quantize``.

    Rotate Q and K of one problem with the same vector, so that Q K^T is
    unchanged; the draw is torch's CPU generator, copied to ``device``.
    """
    g = torch.Generator().manual_seed(int(seed))
    s = torch.randint(0, 2, (int(d),), generator=g, dtype=torch.int8) * 2 - 1
    return s.to(device) if device is not None else s


@_nvtx("fa.fp8_quantize")
def fp8_quantize(x: torch.Tensor, signs: Optional[torch.Tensor] = None, transpose: bool = False,
                 out: Optional[torch.Tensor] = None, descale: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """e4m3 codes of a bf16 tensor with one descale per (batch, head); returns (x8, descale).

    x [B, H, N, d] bf16 on the GPU (d = 64 or 128).  x8 is uint8 [B, H, N, d],
    or [B, H, d, N] with ``transpose`` (the layout ``fwd_fp8`` takes for V;
    N a multiple of 16).  With ``signs`` (int8 [d] of +-1 on the same device,
    see ``hadamard_signs``) each row is rotated by diag(signs) H_d / sqrt(d)
    first: the incoherent processing of the 8-bit path.  code * descale[b, h]
    approximates the (rotated) value.
    """
    _check(x, "x", torch.bfloat16, 4, None)
    dev = x.device
    B, H, N, d = x.shape
    shape = (B, H, d, N) if transpose else (B, H, N, d)
    if out is None:
        out = torch.empty(shape, dtype=torch.uint8, device=dev)
    else:
        _check(out, "out", torch.uint8, 4, dev)
        if tuple(out.shape) != shape:
            raise ValueError("out must be %s" % (shape,))
    if descale is None:
        descale = torch.empty((B, H), dtype=torch.float32, device=dev)
    else:
        _check(descale, "descale", torch.float32, 2, dev)
        if tuple(descale.shape) != (B, H):
            raise ValueError("descale must be %s" % ((B, H),))
    sp = 0
    if signs is not None:
        _check(signs, "signs", torch.int8, 1, dev)
        if signs.numel() != d:
            raise ValueError("signs must have d = %d entries" % d)
        sp = signs.data_ptr()
    with torch.cuda.device(dev):
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        st = fa_fp8_quantize(x.data_ptr(), out.data_ptr(), descale.data_ptr(), B, H, N, d, bool(transpose),
                             sp or None, s.cuda_stream)
    if st != 0:
        raise FaError(st, "fa_fp8_quantize")
    return out, descale


@_nvtx("fa.fwd_fp8_from_bf16")
def fwd_fp8_from_bf16(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                      scale: Optional[float] = None, rotate: bool = True, seed: int = 0,
                      stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """The 8-bit forward from bf16 inputs: quantizes Q and K (rotated with one
    seeded sign vector when ``rotate``) and V (transposed), then runs
    ``fwd_fp8``; returns (O bf16, LSE fp32).  Dense layout, d = 64 or 128."""
    signs = hadamard_signs(q.shape[-1], seed, q.device) if rotate else None
    q8, qd = fp8_quantize(q, signs, stream=stream)
    k8, kd = fp8_quantize(k, signs, stream=stream)
    vt8, vd = fp8_quantize(v, None, transpose=True, stream=stream)
    return fwd_fp8(q8, k8, vt8, qd, kd, vd, causal=causal, scale=scale, stream=stream)
