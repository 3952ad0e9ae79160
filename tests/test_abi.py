"""The C-ABI library on the CPU side: it builds, loads, exports every symbol
include/gqa_attn.h declares, and its host-side argument checks return the
documented status before anything reaches a GPU."""
import ctypes
import os
import re

import pytest

from gqa_softmax_attention_gb300 import _lib, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gqa_attn.h")
OK, INVALID, UNSUPPORTED, MISALIGNED, WORKSPACE = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\**\s+\**\s*([A-Za-z_]\w*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("attn_fwd_dense", "attn_decode_paged", "attn_decode_paged_workspace_size", "attn_validate_paged",
              "attn_fwd_varlen", "attn_fwd_paged", "attn_varlen_workspace_size", "attn_paged_workspace_size",
              "attn_decode_paged_fp8kv",
              "gqa_status_string", "gqa_device_error", "gqa_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(7):
        assert lib.gqa_status_string(code)
    assert b"sm_103a" in lib.gqa_version()


A16 = ctypes.c_void_p(1 << 20)         # 16-byte aligned stand-in pointers; never dereferenced
A16b = ctypes.c_void_p(2 << 20)
MIS = ctypes.c_void_p((1 << 20) + 2)   # misaligned


def dense(lib, q=A16, k=A16, v=A16, o=A16b, B=1, Hq=4, Hkv=2, Sq=8, Skv=8, D=64, scale=0.125, lse=None):
    return lib.attn_fwd_dense(q, k, v, None, o, lse, B, Hq, Hkv, Sq, Skv, D, 1, scale, None)


def test_dense_argument_checks(lib):
    assert dense(lib, B=0) == INVALID
    assert dense(lib, Hq=6, Hkv=4) == INVALID                   # Hq % Hkv != 0
    assert dense(lib, Sq=-1) == INVALID
    assert dense(lib, Skv=-3) == INVALID
    assert dense(lib, D=96) == UNSUPPORTED
    assert dense(lib, D=512) == UNSUPPORTED
    assert dense(lib, scale=float("nan")) == INVALID
    assert dense(lib, scale=float("inf")) == INVALID
    assert dense(lib, q=MIS) == MISALIGNED
    assert dense(lib, o=MIS) == MISALIGNED
    assert dense(lib, lse=ctypes.c_void_p((1 << 20) + 1)) == MISALIGNED
    assert dense(lib, q=None) == INVALID
    assert dense(lib, Sq=0) == OK                                # nothing to do, nothing launched


def paged(lib, ws=None, ws_bytes=0, q=A16, B=2, Sq=1, Hq=8, Hkv=2, D=128, ps=16, num_pages=10, max_pages=4,
          seq=A16, table=A16):
    return lib.attn_decode_paged(q, A16, A16, seq, table, ps, A16b, None, B, Sq, Hq, Hkv, D, num_pages, max_pages,
                                 1, 0.1, ws, ws_bytes, None)


def test_paged_argument_checks(lib):
    assert paged(lib, B=0) == INVALID
    assert paged(lib, Hq=6, Hkv=4) == INVALID
    assert paged(lib, ps=0) == INVALID
    assert paged(lib, max_pages=0) == INVALID
    assert paged(lib, D=80) == UNSUPPORTED
    assert paged(lib, q=MIS) == MISALIGNED
    assert paged(lib, seq=ctypes.c_void_p((1 << 20) + 2)) == MISALIGNED
    assert paged(lib, ws=None, ws_bytes=0) == WORKSPACE          # workspace is required
    assert paged(lib, ws=A16, ws_bytes=16) == WORKSPACE          # and must be large enough
    assert paged(lib, Sq=0) == OK


def paged_fp8(lib, ws=None, ws_bytes=0, q=A16, kc=A16, ks=None, vs=None, B=2, Sq=1, Hq=8, Hkv=2, D=128, ps=16,
              num_pages=10, max_pages=4):
    return lib.attn_decode_paged_fp8kv(q, kc, A16, ks, vs, A16, A16, ps, A16b, None, B, Sq, Hq, Hkv, D, num_pages,
                                       max_pages, 1, 0.1, None, ws, ws_bytes, None)


def test_paged_fp8kv_argument_checks(lib):
    assert paged_fp8(lib, B=0) == INVALID
    assert paged_fp8(lib, Hq=6, Hkv=4) == INVALID
    assert paged_fp8(lib, D=64) == UNSUPPORTED                  # e4m3 rows of 128 or 256 bytes only
    assert paged_fp8(lib, kc=MIS) == MISALIGNED
    assert paged_fp8(lib, ks=ctypes.c_void_p((1 << 20) + 2)) == MISALIGNED
    assert paged_fp8(lib, ws=None, ws_bytes=0) == WORKSPACE
    assert paged_fp8(lib, ws=A16, ws_bytes=16) == WORKSPACE
    assert paged_fp8(lib, Sq=0) == OK


def varlen(lib, q=A16, o=A16b, cu=A16, cukv=A16, B=2, total_q=8, total_kv=16, Hq=4, Hkv=2, D=64, ws=A16,
           ws_bytes=1 << 20, opts=None):
    return lib.attn_fwd_varlen(q, A16, A16, cu, cukv, o, None, B, total_q, total_kv, Hq, Hkv, D, 1, 0.125, opts, ws,
                               ws_bytes, None)


def paged_varlen(lib, q=A16, cu=A16, B=2, total_q=8, Hq=4, Hkv=2, D=64, ps=16, num_pages=4, max_pages=2, ws=A16,
                 ws_bytes=1 << 20):
    return lib.attn_fwd_paged(q, A16, A16, cu, A16, A16, ps, A16b, None, B, total_q, Hq, Hkv, D, num_pages, max_pages,
                              1, 0.125, None, ws, ws_bytes, None)


def test_varlen_argument_checks(lib):
    # TileOPs GQAVarlenFwdOp / GQAPagedFwdOp: refused before anything is launched
    assert varlen(lib, B=0) == INVALID
    assert varlen(lib, Hq=6, Hkv=4) == INVALID
    assert varlen(lib, total_q=-1) == INVALID
    assert varlen(lib, D=96) == UNSUPPORTED
    assert varlen(lib, Hq=258, Hkv=1) == UNSUPPORTED              # more than 128 heads per KV head
    assert varlen(lib, q=MIS) == MISALIGNED
    assert varlen(lib, cu=ctypes.c_void_p((1 << 20) + 2)) == MISALIGNED
    assert varlen(lib, cu=None) == INVALID
    assert varlen(lib, ws=None, ws_bytes=0) == WORKSPACE
    assert varlen(lib, ws_bytes=lib.attn_varlen_workspace_size(2, 8, 4, 2) - 1) == WORKSPACE
    assert varlen(lib, ws=ctypes.c_void_p((1 << 20) + 8)) == MISALIGNED
    assert varlen(lib, total_q=0) == OK                          # nothing to do, nothing launched
    assert paged_varlen(lib, ps=0) == INVALID
    assert paged_varlen(lib, num_pages=0) == INVALID
    assert paged_varlen(lib, D=80) == UNSUPPORTED
    assert paged_varlen(lib, ws=None, ws_bytes=0) == WORKSPACE
    assert paged_varlen(lib, total_q=0) == OK
    # workspace: a header and two 32-byte entries per possible row block
    assert lib.attn_varlen_workspace_size(2, 8, 4, 2) == 16 + 64 * (8 // 64 + 2 + 1)
    assert lib.attn_varlen_workspace_size(3, 1000, 24, 2) == 16 + 64 * (1000 // 10 + 3 + 1)   # g = 12: 10 queries
    assert lib.attn_varlen_workspace_size(2, 8, 6, 4) == 0


def test_paged_workspace_holds_the_decode_partials(lib):
    """attn_fwd_paged's larger workspace: the packed plan's bytes, a 256-byte
    boundary, then attn_decode_paged's workspace for B one-query requests; the
    packed size alone when the group is too wide for the split decode kernel."""
    for B, tq, Hq, Hkv, D, ps, mp in ((64, 4156, 32, 8, 128, 64, 257), (3, 10, 24, 2, 256, 16, 40)):
        v = lib.attn_varlen_workspace_size(B, tq, Hq, Hkv)
        d = lib.attn_decode_paged_workspace_size(B, 1, Hq, Hkv, D, ps, mp)
        assert lib.attn_paged_workspace_size(B, tq, Hq, Hkv, D, ps, mp) == (v + 255) // 256 * 256 + d
    # 64 query heads per KV head: the decode rows would take the tensor-core kernel
    assert lib.attn_paged_workspace_size(4, 8, 64, 1, 128, 64, 8) == lib.attn_varlen_workspace_size(4, 8, 64, 1)
    assert lib.attn_paged_workspace_size(2, 8, 6, 4, 128, 64, 8) == 0


def test_workspace_size_is_positive_and_monotone(lib):
    small = lib.attn_decode_paged_workspace_size(4, 1, 32, 8, 128, 64, 16)
    big = lib.attn_decode_paged_workspace_size(64, 1, 32, 8, 128, 64, 256)
    assert 0 < small < big
    assert lib.attn_decode_paged_workspace_size(4, 1, 30, 8, 128, 64, 16) == 0   # Hq % Hkv
    assert lib.attn_decode_paged_workspace_size(4, 1, 32, 8, 96, 64, 16) == 0    # D


def test_python_layer_rejects_cpu_tensors():
    import torch
    import gqa_softmax_attention_gb300 as g
    q = torch.zeros(1, 4, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        g.attention(q, q, q)


class Opts(ctypes.Structure):
    _fields_ = [("window_left", ctypes.c_int), ("window_right", ctypes.c_int), ("softcap", ctypes.c_float),
                ("sinks", ctypes.c_void_p), ("dtype", ctypes.c_int)]


def test_option_checks(lib):
    # refused before anything is launched (TileOPs GQADenseFwdOp: window -1 = unlimited, softcap >= 0)
    def dense_ex(o):
        return lib.attn_fwd_dense_ex(A16, A16, A16, None, A16b, None, 1, 4, 2, 8, 8, 64, 1, 0.125, ctypes.byref(o),
                                     None)

    def paged_ex(o):
        return lib.attn_decode_paged_ex(A16, A16, A16, A16, A16, 16, A16b, None, 2, 1, 8, 2, 128, 10, 4, 1, 0.1,
                                        ctypes.byref(o), A16, 1 << 30, None)

    for call in (dense_ex, paged_ex):
        assert call(Opts(-2, -1, 0.0, None)) == INVALID
        assert call(Opts(-1, -5, 0.0, None)) == INVALID
        assert call(Opts(-1, -1, -1.0, None)) == INVALID
        assert call(Opts(-1, -1, float("nan"), None)) == INVALID
        assert call(Opts(-1, -1, float("inf"), None)) == INVALID
        assert call(Opts(-1, -1, 0.0, (1 << 20) + 2)) == MISALIGNED
        assert call(Opts(-1, -1, 0.0, None, 2)) == INVALID       # neither GQA_BF16 nor GQA_FP16


def test_python_layer_option_checks():
    import torch
    import gqa_softmax_attention_gb300.api as api
    with pytest.raises(ValueError, match="window_left"):
        api._options(-3, -1, None, None, 4, "cpu")
    with pytest.raises(ValueError, match="softcap"):
        api._options(-1, -1, -0.5, None, 4, "cpu")
    with pytest.raises(ValueError, match="sinks"):
        api._options(-1, -1, None, torch.zeros(3), 4, "cpu")
    assert api._options(-1, -1, None, None, 4, "cpu") == (None, None)
