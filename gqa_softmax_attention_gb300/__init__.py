"""GB300-native causal grouped-query softmax attention forward (sm_103a).

Dense prefill, paged decode (16-bit or float8_e4m3fn key/value caches) and
packed variable-length calls (dense, or mixed prefill and decode over a paged
cache), bf16 or fp16 in / FP32 accumulation / 16-bit out, with an FP32
natural-log log-sum-exp per row.  Every step runs in
this package's CUDA kernels behind a C ABI (``include/gqa_attn.h``); this
Python layer only marshals arguments.  The shared library is loaded on first use and its absence
is an error: there is no CPU fallback.
"""

from .api import (attention, attn_decode_paged, attn_decode_paged_fp8kv, attn_decode_paged_noalloc,  # noqa: F401
                  attn_decode_paged_workspace_size, attn_fwd_paged, attn_fwd_varlen,
                  attn_fwd_dense, attn_paged_workspace_size, attn_validate_paged, attn_varlen_workspace_size,
                  decode_paged,
                  gqa_device_error, paged, resolve_scale, varlen)
