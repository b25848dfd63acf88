"""GB300-native exact attention forward (FlashAttention-style, sm_103a).

``fwd`` runs the library's tcgen05 kernel through the C ABI in ``libfa.so``
(declared in ``include/fa.h``).  There is no CPU fallback: if the library is
not built, or no sm_103 GPU is present, the call raises.
"""
from ._lib import (FaError, fa_fwd, fa_decode, fa_status_string, fa_device_status, fa_fwd_smem_bytes,  # noqa: F401
                   fa_fwd_threads, fa_debug_fault_injection, fa_debug_exp2_soft, lib)
from .api import fwd, fwd_host  # noqa: F401
from .build import build, LIB_PATH  # noqa: F401
