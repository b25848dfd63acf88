"""GB300-native exact attention (FlashAttention-style, sm_103a).

``fwd`` and ``bwd`` run the library's tcgen05 kernels through the C ABI in ``libfa.so``
(declared in ``include/fa.h``).  There is no CPU fallback: if the library is
not built, or no sm_103 GPU is present, the call raises.
"""
from ._lib import (FaError, fa_fwd, fa_fwd_host, fa_decode, fa_bwd, fa_fwd_fp8, fa_fp8_quantize, fa_status_string,  # noqa: F401
                   fa_device_status, fa_fwd_smem_bytes, fa_fwd_threads, fa_bwd_smem_bytes, fa_debug_fault_injection,
                   fa_debug_exp2_soft, fa_debug_soft_exp, fa_debug_fwd_pair, fa_debug_schedule, lib, lib_path)
from .api import bwd, fp8_quantize, fwd, fwd_fp8, fwd_fp8_from_bf16, fwd_host, hadamard_signs  # noqa: F401
from .build import build, LIB_PATH  # noqa: F401
