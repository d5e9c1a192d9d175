"""GB300 (sm_103a) tiled FlashAttention forward.

The computation runs in hand-written CUDA kernels behind the C ABI of
libfa_fwd.so (include/fa_fwd.h).  This package is the Python binding: the
same entry points, argument marshalling only (torch tensors -> device
pointers, the current torch stream).  There is no fallback: without the
library every call raises.
"""
from ._binding import (  # noqa: F401
    FA_ERR_ALIGN, FA_ERR_CUDA, FA_ERR_DEVICE_TIMEOUT, FA_ERR_NULL, FA_ERR_RANGE, FA_ERR_SCRATCH,
    FA_ERR_SHAPE, FA_ERR_THRESHOLD, FA_ERR_UNSUPPORTED, FA_OK,
    FA_DTYPE_FP16, FA_FP8_E4M3, FA_FP8_E5M2, FA_MASK_CAUSAL, FA_MASK_CAUSAL_DIAG_BLOCK, FA_MASK_NONE, FA_V_FP16,
    FA_V_FROM_K, FaError, fa_bwd, fa_check_status, fa_convert_v_fp16, fa_fwd, fa_fwd_noalloc,
    fa_fwd_ext, fa_fwd_fp8, fa_fwd_o_lo, fa_extras_t, fa_set_max_kv_split, fa_set_wait_timeout_ns, fa_strerror, fa_wait_probe,
    flash_attention_backward, flash_attention_forward, flash_attention_forward_fp8, library, library_path,
)
