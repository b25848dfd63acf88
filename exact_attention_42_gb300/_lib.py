"""ctypes binding of libfa.so: the C-ABI entry points, same names, no logic."""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH

FA_OK = 0
STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_NULL", 2: "FA_ERR_SHAPE", 3: "FA_ERR_ALIGN", 4: "FA_ERR_UNSUPPORTED",
                5: "FA_ERR_CUDA", 6: "FA_ERR_TIMEOUT", 7: "FA_ERR_VALUE"}

_lib = None
_lock = threading.Lock()


class FaError(RuntimeError):
    """A non-zero fa_status returned by the library."""

    def __init__(self, status: int, what: str = "fa_fwd"):
        self.status = status
        super().__init__("%s failed: %s" % (what, fa_status_string(status)))


def lib_path() -> str:
    """The library this process loads: libfa.so, or the one FA_LIBRARY names
    (the debug build's tests point it at libfa_debug.so)."""
    return os.environ.get("FA_LIBRARY") or LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                raise RuntimeError("%s is not built; run exact_attention_42_gb300.build.build()" % path)
            L = ctypes.CDLL(path)
            vp, ci = ctypes.c_void_p, ctypes.c_int
            L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ctypes.c_float, ci, vp, vp]
            L.fa_fwd.restype = ci
            L.fa_status_string.argtypes = [ci]
            L.fa_status_string.restype = ctypes.c_char_p
            L.fa_device_status.argtypes = [ctypes.POINTER(ci)]
            L.fa_device_status.restype = ci
            L.fa_fwd_smem_bytes.argtypes = [ci]
            L.fa_fwd_smem_bytes.restype = ci
            L.fa_fwd_threads.argtypes = []
            L.fa_fwd_threads.restype = ci
            L.fa_debug_fault_injection.argtypes = [ci, ctypes.c_double]
            L.fa_debug_fault_injection.restype = ci
            L.fa_debug_fwd_pair.argtypes = [ci]
            L.fa_debug_fwd_pair.restype = ci
            L.fa_debug_soft_exp.argtypes = [ci]
            L.fa_debug_soft_exp.restype = ci
            L.fa_debug_exp2_soft.argtypes = [vp, vp, ci, vp]
            L.fa_debug_exp2_soft.restype = ci
            L.fa_decode.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ctypes.c_float, ci, vp]
            L.fa_decode.restype = ci
            L.fa_decode_smem_bytes.argtypes = [ci]
            L.fa_decode_smem_bytes.restype = ci
            L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ctypes.c_float, ci,
                                 vp, vp]
            L.fa_bwd.restype = ci
            L.fa_fwd_fp8.argtypes = [vp] * 8 + [ci] * 6 + [ctypes.c_float, ci, vp, vp]
            L.fa_fwd_fp8.restype = ci
            L.fa_bwd_smem_bytes.argtypes = [ci]
            L.fa_bwd_smem_bytes.restype = ci
            L.fa_fp8_quantize.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, vp, vp]
            L.fa_fp8_quantize.restype = ci
            L.fa_fwd_host.argtypes = [vp] * 10 + [ci] * 6 + [ctypes.c_float, ci, vp, vp, ci, vp]
            L.fa_fwd_host.restype = ci
            L.fa_debug_schedule.argtypes = [ci] * 9 + [vp, vp, ci, ctypes.POINTER(ci)]
            L.fa_debug_schedule.restype = ci
            _lib = L
    return _lib


def fa_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, cu_seqlens, stream) -> int:
    """Direct call of the C entry point with integer addresses; returns the status."""
    return lib().fa_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, ctypes.c_float(scale), int(causal),
                        cu_seqlens, stream)


def fa_fwd_host(q_h, k_h, v_h, o_h, lse_h, q_d, k_d, v_d, o_d, lse_d, B, Hq, Hkv, Nq, Nk, d, scale, causal,
                cu_h, cu_d, pieces, stream) -> int:
    """Direct call of the host-buffer forward with integer addresses; returns the status."""
    return lib().fa_fwd_host(q_h, k_h, v_h, o_h, lse_h, q_d, k_d, v_d, o_d, lse_d, B, Hq, Hkv, Nq, Nk, d,
                             ctypes.c_float(scale), int(causal), cu_h, cu_d, int(pieces), stream)


def fa_decode(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, stream) -> int:
    """Direct call of the split-KV entry point with integer addresses; returns the status."""
    return lib().fa_decode(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, ctypes.c_float(scale), int(causal), stream)


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, delta, B, Hq, Hkv, Nq, Nk, d, scale, causal, cu_seqlens,
           stream) -> int:
    """Direct call of the backward entry point with integer addresses; returns the status."""
    return lib().fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, delta, B, Hq, Hkv, Nq, Nk, d, ctypes.c_float(scale),
                        int(causal), cu_seqlens, stream)


def fa_fwd_fp8(q8, k8, vt8, q_descale, k_descale, v_descale, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal,
               cu_seqlens, stream) -> int:
    """Direct call of the 8-bit forward entry point with integer addresses; returns the status."""
    return lib().fa_fwd_fp8(q8, k8, vt8, q_descale, k_descale, v_descale, o, lse, B, Hq, Hkv, Nq, Nk, d,
                            ctypes.c_float(scale), int(causal), cu_seqlens, stream)


def fa_fp8_quantize(x, x8, descale, B, H, N, d, transpose, signs, stream) -> int:
    """Direct call of the e4m3 quantization entry point with integer addresses; returns the status."""
    return lib().fa_fp8_quantize(x, x8, descale, B, H, N, d, int(transpose), signs, stream)


def fa_status_string(status: int) -> str:
    try:
        return lib().fa_status_string(int(status)).decode()
    except RuntimeError:
        return STATUS_NAMES.get(int(status), "unknown status %d" % status)


def fa_device_status() -> int:
    """Reads and clears the device status words (waits for all work on the device first)."""
    bits = ctypes.c_int(0)
    st = lib().fa_device_status(ctypes.byref(bits))
    if st not in (0, 6):
        raise FaError(st, "fa_device_status")
    return bits.value


def fa_debug_fault_injection(mode: int, wait_limit_seconds: float = 0.0) -> None:
    """Test hook: modes 1-4 make one kernel's later launches time out on purpose (see fa.h)."""
    st = lib().fa_debug_fault_injection(int(mode), float(wait_limit_seconds))
    if st != 0:
        raise FaError(st, "fa_debug_fault_injection")


def fa_debug_soft_exp(on: int) -> None:
    """Test hook: 1 selects the forward kernels with software exponentials (see fa.h)."""
    st = lib().fa_debug_soft_exp(int(on))
    if st != 0:
        raise FaError(st, "fa_debug_soft_exp")


def fa_debug_fwd_pair(on: int) -> None:
    """Test hook: 1 selects the CTA-pair forward kernel for bf16, d = 128 (see fa.h)."""
    st = lib().fa_debug_fwd_pair(int(on))
    if st != 0:
        raise FaError(st, "fa_debug_fwd_pair")


def fa_debug_schedule(kernel: int, B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int, causal: bool,
                      workers: int):
    """The worker lists a persistent launch would run (see fa.h): a list of unit
    lists, one per worker, or None when the kernel uses its built-in order."""
    cap = 1 << 16
    start = (ctypes.c_int32 * (workers + 1))()
    units = (ctypes.c_int32 * cap)()
    n = ctypes.c_int(0)
    st = lib().fa_debug_schedule(int(kernel), B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), workers,
                                 ctypes.cast(start, ctypes.c_void_p), ctypes.cast(units, ctypes.c_void_p), cap,
                                 ctypes.byref(n))
    if st != 0:
        raise FaError(st, "fa_debug_schedule")
    if n.value == 0:
        return None
    return [list(units[start[w]:start[w + 1]]) for w in range(n.value)]


def fa_debug_exp2_soft(x_ptr: int, y_ptr: int, n: int, stream: int = 0) -> None:
    """Test entry point: the kernel's software 2^x on n device floats."""
    st = lib().fa_debug_exp2_soft(x_ptr, y_ptr, int(n), stream)
    if st != 0:
        raise FaError(st, "fa_debug_exp2_soft")


def fa_fwd_smem_bytes(d: int) -> int:
    return lib().fa_fwd_smem_bytes(d)


def fa_fwd_threads() -> int:
    return lib().fa_fwd_threads()


def fa_bwd_smem_bytes(d: int) -> int:
    return lib().fa_bwd_smem_bytes(d)
