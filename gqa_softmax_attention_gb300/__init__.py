"""GB300-native causal grouped-query softmax attention forward (sm_103a).

Dense prefill and paged decode, bf16 in / FP32 accumulation / bf16 out, with an
FP32 natural-log log-sum-exp per row.  Every step runs in this package's CUDA
kernels behind a C ABI (``include/gqa_attn.h``); this Python layer only
marshals arguments.  The shared library is loaded on first use and its absence
is an error: there is no CPU fallback.
"""

from .api import (attention, attn_decode_paged, attn_decode_paged_noalloc,  # noqa: F401
                  attn_decode_paged_workspace_size,
                  attn_fwd_dense, attn_validate_paged, decode_paged, gqa_device_error,
                  resolve_scale)
