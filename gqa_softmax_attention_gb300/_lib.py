"""ctypes binding of libgqa_attn.so (declared in include/gqa_attn.h).

Loading never falls back to anything: if the library has not been built, the
first call raises.  Build it with ``gqa_softmax_attention_gb300.build.build()``
(``__graft_entry__.build()`` does this).
"""
import ctypes
import os

from . import build as _build

STATUS = {
    0: "GQA_OK",
    1: "GQA_ERR_INVALID_ARG",
    2: "GQA_ERR_UNSUPPORTED",
    3: "GQA_ERR_MISALIGNED",
    4: "GQA_ERR_WORKSPACE",
    5: "GQA_ERR_CUDA",
    6: "GQA_ERR_TIMEOUT",
}

_handle = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libgqa_attn.so once and declare its C signatures."""
    global _handle
    if _handle is not None:
        return _handle
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError("libgqa_attn.so is not built (%s); run gqa_softmax_attention_gb300.build.build()"
                           % path)
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.attn_fwd_dense.argtypes = [vp, vp, vp, vp, vp, vp] + [i] * 7 + [f, vp]
    lib.attn_fwd_dense.restype = i
    lib.attn_decode_paged.argtypes = [vp, vp, vp, vp, vp, i, vp, vp] + [i] * 8 + [f, vp, sz, vp]
    lib.attn_decode_paged.restype = i
    lib.attn_fwd_dense_ex.argtypes = [vp, vp, vp, vp, vp, vp] + [i] * 7 + [f, vp, vp]
    lib.attn_fwd_dense_ex.restype = i
    lib.attn_decode_paged_ex.argtypes = [vp, vp, vp, vp, vp, i, vp, vp] + [i] * 8 + [f, vp, vp, sz, vp]
    lib.attn_decode_paged_ex.restype = i
    lib.attn_decode_paged_fp8kv.argtypes = [vp] * 7 + [i, vp, vp] + [i] * 8 + [f, vp, vp, sz, vp]
    lib.attn_decode_paged_fp8kv.restype = i
    lib.attn_decode_paged_workspace_size.argtypes = [i] * 7
    lib.attn_decode_paged_workspace_size.restype = sz
    lib.attn_decode_paged_noalloc.argtypes = [vp, vp, vp, vp, vp, i, vp, vp] + [i] * 8 + [f, vp]
    lib.attn_decode_paged_noalloc.restype = i
    lib.attn_decode_paged_noalloc_max_workspace.argtypes = []
    lib.attn_decode_paged_noalloc_max_workspace.restype = sz
    lib.attn_fwd_varlen.argtypes = [vp] * 7 + [i] * 7 + [f, vp, vp, sz, vp]
    lib.attn_fwd_varlen.restype = i
    lib.attn_fwd_paged.argtypes = [vp] * 6 + [i, vp, vp] + [i] * 8 + [f, vp, vp, sz, vp]
    lib.attn_fwd_paged.restype = i
    lib.attn_varlen_workspace_size.argtypes = [i] * 4
    lib.attn_varlen_workspace_size.restype = sz
    lib.attn_paged_workspace_size.argtypes = [i] * 7
    lib.attn_paged_workspace_size.restype = sz
    lib.attn_validate_paged.argtypes = [vp, vp] + [i] * 6 + [vp]
    lib.attn_validate_paged.restype = i
    lib.gqa_status_string.argtypes = [i]
    lib.gqa_status_string.restype = ctypes.c_char_p
    lib.gqa_device_error.argtypes = []
    lib.gqa_device_error.restype = i
    lib.gqa_version.argtypes = []
    lib.gqa_version.restype = ctypes.c_char_p
    _handle = lib
    return lib


class Options(ctypes.Structure):
    """gqa_options of include/gqa_attn.h."""
    _fields_ = [("window_left", ctypes.c_int), ("window_right", ctypes.c_int), ("softcap", ctypes.c_float),
                ("sinks", ctypes.c_void_p), ("dtype", ctypes.c_int)]


def status_name(code: int) -> str:
    return STATUS.get(code, "status %d" % code)
