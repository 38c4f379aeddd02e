"""exact_io_aware_21_gb300: exact IO-aware attention (FlashAttention) for GB300 (sm_103a).

The compute path is a C-ABI CUDA library (``libfa_gb300.so``, header
``include/fa.h``); this package is its thin Python binding.  The library is
loaded on first use and every op raises if it is missing: there is no CPU
fallback.
"""

from .binding import (  # noqa: F401
    FAError,
    fa_bwd,
    fa_decode,
    fa_decode_paged,
    fa_fwd,
    fa_fwd_fp8,
    fa_quantize_fp8,
    forward,
    forward_fp8,
    forward_varlen,
    forward_blocksparse,
    backward_blocksparse,
    fa_bwd_blocksparse,
    fa_fwd_blocksparse,
    backward_varlen,
    fa_fwd_varlen,
    fa_bwd_varlen,
    quantize_fp8,
    backward,
    decode,
    decode_paged,
    library,
    library_path,
)
