"""GB300 (sm_103a) fused attention forward with the online-softmax recurrence.

The computation lives in ``libattn.so`` (CUDA sources under ``csrc/``, C ABI in
``include/attn.h``); this package only binds it. Build it with
``python -m online_softmax_fwd_gb300.build``.
"""
from ._binding import (P_SCALE_BLOCK_AMAX, P_SCALE_CONSTANT, P_SCALE_CONSTANT_E5M2, AttnError, Status, attn_bwd,
                       attn_bwd_mxfp8, attn_combine, attn_fwd, attn_fwd_2cta, attn_fwd_from_host, attn_fwd_mxfp8, attn_fwd_raw, attn_fwd_rescale_log,
                       device_status,                        exp2_emulated, lib, mxfp8_quantize, mxfp8_scale_bytes, status_string, version)

__all__ = ["P_SCALE_BLOCK_AMAX", "P_SCALE_CONSTANT", "P_SCALE_CONSTANT_E5M2", "AttnError", "Status", "attn_bwd",
           "attn_bwd_mxfp8", "attn_combine", "attn_fwd", "attn_fwd_2cta", "attn_fwd_from_host", "attn_fwd_mxfp8", "attn_fwd_raw", "attn_fwd_rescale_log",
           "device_status",
           "exp2_emulated", "lib", "mxfp8_quantize", "mxfp8_scale_bytes", "status_string", "version"]
