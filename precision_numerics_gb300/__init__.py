"""GB300-native (sm_103a) exact tiled attention: BF16 forward and backward.

The compute path is the CUDA library libattn.so (C ABI, include/attn.h);
`precision_numerics_gb300.attn` is its thin Python binding.
"""
from .attn import (AttnError, attn_bwd, attn_bwd_dq_convert, attn_bwd_main,  # noqa: F401
                   attn_bwd_preprocess, attn_bwd_workspace_bytes, attn_check_status, attn_fwd,
                   attn_fwd_stable, attn_bwd_noalloc, attn_quantize_int8, attn_fwd_int8,
                   attn_quantize_int8_as_bf16, attn_fwd_int8_as_bf16, int8_scale_rows,
                   attn_selftest_wait_timeout, attn_version, load_library)

__all__ = ["AttnError", "attn_fwd", "attn_fwd_stable", "attn_quantize_int8", "attn_fwd_int8",
           "attn_quantize_int8_as_bf16", "attn_fwd_int8_as_bf16", "int8_scale_rows",
           "attn_bwd", "attn_bwd_noalloc", "attn_bwd_preprocess", "attn_bwd_main",
           "attn_bwd_dq_convert", "attn_bwd_workspace_bytes", "attn_check_status",
           "attn_selftest_wait_timeout", "attn_version", "load_library"]
