"""FP64 CPU oracle for causal grouped-query softmax attention forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference arm may import this package.  It shares
no code with the CUDA library and the product path never calls it.

The arithmetic lives in ``oracle_fp64.c`` (plain C, double precision, one row
at a time); this module only marshals arrays.  Inputs may be torch tensors
(bfloat16, float16, float32 or float64, any device-less CPU tensor) or numpy
arrays; 16- and 32-bit values widen to double exactly.  Outputs are float64
torch tensors: ``o`` shaped like ``q`` and ``lse`` shaped ``q.shape[:-1]``.

Parity status: every function here is pinned by ``tests/test_oracle.py``.
"""
import ctypes
import math

import numpy as np
import torch

from . import build as _build

_F64, _BF16, _F16 = 0, 1, 2


def _bind(lib):
    vp, ip = ctypes.c_void_p, ctypes.c_int
    lib.oracle_attn_dense.argtypes = [vp] * 3 + [ip] + [vp] * 3 + [ip] * 7 + [ctypes.c_double, ip]
    lib.oracle_attn_dense.restype = ip
    lib.oracle_attn_dense_rows.argtypes = ([vp] * 3 + [ip] + [vp] * 2 + [ip] + [vp] * 2 + [ip] * 7
                                           + [ctypes.c_double, ip])
    lib.oracle_attn_dense_rows.restype = ip
    lib.oracle_attn_paged.argtypes = ([vp] * 3 + [ip] + [vp] * 2 + [ip] + [vp] * 3 + [ip] * 8
                                      + [ctypes.c_double, ip])
    lib.oracle_attn_paged.restype = ip
    lp, dp = ctypes.c_long, ctypes.c_double
    lib.oracle_attn_dense_ex.argtypes = ([vp] * 3 + [ip] + [vp] * 3 + [ip] * 7 + [dp, lp, lp, dp, vp, ip])
    lib.oracle_attn_dense_ex.restype = ip
    lib.oracle_attn_dense_rows_ex.argtypes = ([vp] * 3 + [ip] + [vp] * 2 + [ip] + [vp] * 2 + [ip] * 7
                                              + [dp, lp, lp, dp, vp, ip])
    lib.oracle_attn_dense_rows_ex.restype = ip
    lib.oracle_attn_paged_ex.argtypes = ([vp] * 3 + [ip] + [vp] * 2 + [ip] + [vp] * 3 + [ip] * 8
                                         + [dp, lp, lp, dp, vp, ip])
    lib.oracle_attn_paged_ex.restype = ip
    lib.oracle_attn_varlen_ex.argtypes = ([vp] * 3 + [ip] + [vp] * 4 + [ip] * 7 + [dp, lp, lp, dp, vp, ip])
    lib.oracle_attn_varlen_ex.restype = ip
    lib.oracle_attn_paged_varlen_ex.argtypes = ([vp] * 3 + [ip] + [vp] * 3 + [ip] + [vp] * 2 + [ip] * 8
                                                + [dp, lp, lp, dp, vp, ip])
    lib.oracle_attn_paged_varlen_ex.restype = ip
    lib.oracle_e4m3_decode.argtypes = [vp, vp, lp]
    lib.oracle_e4m3_decode.restype = ip
    lib.oracle_attn_paged_fp8kv_ex.argtypes = ([vp, ip] + [vp] * 6 + [ip] + [vp] * 3 + [ip] * 8
                                               + [dp, lp, lp, dp, vp, ip])
    lib.oracle_attn_paged_fp8kv_ex.restype = ip
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ip
    return lib


_lib = None


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(_build.build()))
    return _lib


class use_library:
    """Route every call, for the duration of a ``with`` block, to another build
    of ``oracle_fp64.c`` at ``path``.  Tests use it to plant a mistake in a copy
    of the oracle and check that the pins catch it."""

    def __init__(self, path):
        self.lib = _bind(ctypes.CDLL(path))
        self.prev = None

    def __enter__(self):
        global _lib
        self.prev = _load()
        _lib = self.lib
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.prev
        return False


def max_threads() -> int:
    """Threads the oracle's parallel loops use (1 if built without OpenMP)."""
    return _load().oracle_max_threads()


_ERRORS = {
    -1: "bad size argument",
    -2: "Hq must be divisible by Hkv",
    -3: "out of host memory",
    -4: "row index out of range",
    -5: "a request length lies outside [0, max_pages * page_size]",
    -6: "a block_table entry for a used page lies outside [0, num_pages)",
    -7: "a window size below -1",
    -8: "softcap must be finite and >= 0",
    -9: "cu_seqlens must run from 0 up to the packed total without decreasing",
}


def _check(rc):
    if rc != 0:
        raise ValueError("oracle: " + _ERRORS.get(rc, "error %d" % rc))


def _tensor_in(x):
    """Return (numpy array kept alive, dtype code) for a q/k/v-like input."""
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous()
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16), _BF16
        if x.dtype == torch.float16:
            return x.view(torch.int16).numpy().view(np.uint16), _F16
        return x.to(torch.float64).numpy(), _F64
    a = np.ascontiguousarray(x)
    if a.dtype == np.uint16:
        return a, _BF16
    return np.ascontiguousarray(a, dtype=np.float64), _F64


def _same_kind(arrs):
    kinds = {c for _, c in arrs}
    if len(kinds) != 1:
        # mixed input types: widen everything to double
        return [(np.ascontiguousarray(_to_f64(a, c)), _F64) for a, c in arrs]
    return arrs


def _to_f64(a, code):
    if code == _F64:
        return a
    if code == _F16:
        return a.view(np.float16).astype(np.float64)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _mask_in(mask):
    if mask is None:
        return None
    if isinstance(mask, torch.Tensor):
        mask = mask.detach().cpu().contiguous().to(torch.uint8).numpy()
    return np.ascontiguousarray(mask, dtype=np.uint8)


def _opts(window_left, window_right, softcap, sinks, Hq):
    """The optional terms as C arguments: (wl, wr, softcap, sinks array or None)."""
    sk = None
    if sinks is not None:
        sk = np.ascontiguousarray(torch.as_tensor(sinks).detach().cpu().to(torch.float64).numpy().reshape(-1))
        if sk.shape[0] != Hq:
            raise ValueError("oracle: sinks must hold one value per query head")
    return int(window_left), int(window_right), float(0.0 if softcap is None else softcap), sk


def default_scale(D: int) -> float:
    """Scale used when the caller passes None: 1/sqrt(D)."""
    return 1.0 / math.sqrt(D)


def attn_dense(q, k, v, key_padding_mask=None, causal=True, scale=None, nthreads=0,
               window_left=-1, window_right=-1, softcap=0.0, sinks=None):
    """Dense GQA attention in double.  q: [B,Sq,Hq,D]; k, v: [B,Skv,Hkv,D].

    window_left / window_right: keys admitted left / right of the query's key
    position (-1 unlimited); softcap: c > 0 caps each scaled score to
    c*tanh(z/c) (0 or None off); sinks: [Hq] logits added to the softmax
    denominator only, or None."""
    B, Sq, Hq, D = q.shape
    _, Skv, Hkv, _ = k.shape
    if scale is None:
        scale = default_scale(D)
    (qa, c), (ka, _), (va, _) = _same_kind([_tensor_in(q), _tensor_in(k), _tensor_in(v)])
    m = _mask_in(key_padding_mask)
    o = np.zeros((B, Sq, Hq, D), dtype=np.float64)
    lse = np.zeros((B, Sq, Hq), dtype=np.float64)
    wl, wr, cap, sk = _opts(window_left, window_right, softcap, sinks, Hq)
    rc = _load().oracle_attn_dense_ex(_ptr(qa), _ptr(ka), _ptr(va), c, _ptr(m), _ptr(o), _ptr(lse),
                                      B, Hq, Hkv, Sq, Skv, D, int(bool(causal)), float(scale),
                                      wl, wr, cap, _ptr(sk), int(nthreads))
    _check(rc)
    return torch.from_numpy(o), torch.from_numpy(lse)


def attn_dense_rows(q, k, v, rows, key_padding_mask=None, causal=True, scale=None, nthreads=0,
                    window_left=-1, window_right=-1, softcap=0.0, sinks=None):
    """Dense attention for the listed rows only.

    rows: integer array [n, 3] of (b, i, h).  Returns o_rows [n, D], lse_rows [n].
    """
    B, Sq, Hq, D = q.shape
    _, Skv, Hkv, _ = k.shape
    if scale is None:
        scale = default_scale(D)
    (qa, c), (ka, _), (va, _) = _same_kind([_tensor_in(q), _tensor_in(k), _tensor_in(v)])
    m = _mask_in(key_padding_mask)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    n = r.shape[0]
    o = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    wl, wr, cap, sk = _opts(window_left, window_right, softcap, sinks, Hq)
    rc = _load().oracle_attn_dense_rows_ex(_ptr(qa), _ptr(ka), _ptr(va), c, _ptr(m), _ptr(r), n,
                                           _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Skv, D,
                                           int(bool(causal)), float(scale), wl, wr, cap, _ptr(sk),
                                           int(nthreads))
    _check(rc)
    return torch.from_numpy(o), torch.from_numpy(lse)


def attn_paged(q, k_cache, v_cache, real_seqlen_kv, block_table, causal=True, scale=None,
               requests=None, nthreads=0, window_left=-1, window_right=-1, softcap=0.0, sinks=None):
    """Paged GQA attention in double.

    q: [B,Sq,Hq,D]; k_cache, v_cache: [num_pages, page_size, Hkv, D];
    real_seqlen_kv: [B] (query tokens included); block_table: [B, max_pages].
    requests: optional iterable of request indices to compute (others stay 0).
    """
    B, Sq, Hq, D = q.shape
    num_pages, page_size, Hkv, _ = k_cache.shape
    if scale is None:
        scale = default_scale(D)
    (qa, c), (ka, _), (va, _) = _same_kind([_tensor_in(q), _tensor_in(k_cache),
                                            _tensor_in(v_cache)])
    sl = np.ascontiguousarray(torch.as_tensor(real_seqlen_kv).cpu().numpy(), dtype=np.int32)
    bt = np.ascontiguousarray(torch.as_tensor(block_table).cpu().numpy(), dtype=np.int32)
    max_pages = bt.shape[1] if bt.ndim == 2 else 0
    req = None
    if requests is not None:
        req = np.zeros((B,), dtype=np.uint8)
        req[np.asarray(list(requests), dtype=np.int64)] = 1
    o = np.zeros((B, Sq, Hq, D), dtype=np.float64)
    lse = np.zeros((B, Sq, Hq), dtype=np.float64)
    wl, wr, cap, sk = _opts(window_left, window_right, softcap, sinks, Hq)
    rc = _load().oracle_attn_paged_ex(_ptr(qa), _ptr(ka), _ptr(va), c, _ptr(sl), _ptr(bt), page_size,
                                      _ptr(req), _ptr(o), _ptr(lse), B, Sq, Hq, Hkv, D, num_pages,
                                      max_pages, int(bool(causal)), float(scale), wl, wr, cap,
                                      _ptr(sk), int(nthreads))
    _check(rc)
    return torch.from_numpy(o), torch.from_numpy(lse)


def _i32(x):
    return np.ascontiguousarray(torch.as_tensor(x).cpu().numpy(), dtype=np.int32)


def attn_varlen(q, k, v, cu_seqlens_q, cu_seqlens_kv, causal=True, scale=None, nthreads=0,
                window_left=-1, window_right=-1, softcap=0.0, sinks=None):
    """Packed variable-length GQA attention in double (TileOPs GQAVarlenFwdOp).

    q: [total_q, Hq, D]; k, v: [total_kv, Hkv, D]; cu_seqlens_q / cu_seqlens_kv:
    [B + 1] request offsets.  Every request is dense attention over its own rows
    with its own end-aligned causal mask.  Returns o [total_q, Hq, D] and
    lse [total_q, Hq]."""
    total_q, Hq, D = q.shape
    total_kv, Hkv, _ = k.shape
    if scale is None:
        scale = default_scale(D)
    (qa, c), (ka, _), (va, _) = _same_kind([_tensor_in(q), _tensor_in(k), _tensor_in(v)])
    cq, ck = _i32(cu_seqlens_q), _i32(cu_seqlens_kv)
    if cq.shape != ck.shape or cq.ndim != 1 or cq.shape[0] < 1:
        raise ValueError("oracle: cu_seqlens_q and cu_seqlens_kv must both hold B + 1 offsets")
    B = cq.shape[0] - 1
    o = np.zeros((total_q, Hq, D), dtype=np.float64)
    lse = np.zeros((total_q, Hq), dtype=np.float64)
    wl, wr, cap, sk = _opts(window_left, window_right, softcap, sinks, Hq)
    rc = _load().oracle_attn_varlen_ex(_ptr(qa), _ptr(ka), _ptr(va), c, _ptr(cq), _ptr(ck), _ptr(o), _ptr(lse),
                                       B, total_q, total_kv, Hq, Hkv, D, int(bool(causal)), float(scale),
                                       wl, wr, cap, _ptr(sk), int(nthreads))
    _check(rc)
    return torch.from_numpy(o), torch.from_numpy(lse)


def attn_paged_varlen(q, k_cache, v_cache, cu_seqlens_q, cache_seqlens, block_table, causal=True, scale=None,
                      nthreads=0, window_left=-1, window_right=-1, softcap=0.0, sinks=None):
    """Paged GQA attention over packed queries in double (TileOPs GQAPagedFwdOp).

    q: [total_q, Hq, D]; k_cache, v_cache: [num_pages, page_size, Hkv, D];
    cu_seqlens_q: [B + 1]; cache_seqlens: [B] (each request's query tokens
    included); block_table: [B, max_pages].  Returns o [total_q, Hq, D] and
    lse [total_q, Hq]."""
    total_q, Hq, D = q.shape
    num_pages, page_size, Hkv, _ = k_cache.shape
    if scale is None:
        scale = default_scale(D)
    (qa, c), (ka, _), (va, _) = _same_kind([_tensor_in(q), _tensor_in(k_cache), _tensor_in(v_cache)])
    cq, sl, bt = _i32(cu_seqlens_q), _i32(cache_seqlens), _i32(block_table)
    B = sl.shape[0]
    if cq.shape != (B + 1,) or bt.ndim != 2 or bt.shape[0] != B:
        raise ValueError("oracle: cu_seqlens_q [B + 1], cache_seqlens [B] and block_table [B, pages] disagree")
    o = np.zeros((total_q, Hq, D), dtype=np.float64)
    lse = np.zeros((total_q, Hq), dtype=np.float64)
    wl, wr, cap, sk = _opts(window_left, window_right, softcap, sinks, Hq)
    rc = _load().oracle_attn_paged_varlen_ex(_ptr(qa), _ptr(ka), _ptr(va), c, _ptr(cq), _ptr(sl), _ptr(bt),
                                             page_size, _ptr(o), _ptr(lse), B, total_q, Hq, Hkv, D, num_pages,
                                             bt.shape[1], int(bool(causal)), float(scale), wl, wr, cap, _ptr(sk),
                                             int(nthreads))
    _check(rc)
    return torch.from_numpy(o), torch.from_numpy(lse)


def _u8(x):
    """e4m3fn codes (a torch float8_e4m3fn or uint8 tensor, or a numpy array) as uint8."""
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous()
        if x.dtype != torch.uint8:
            x = x.view(torch.uint8)
        return x.numpy()
    return np.ascontiguousarray(x, dtype=np.uint8)


def e4m3_decode(codes):
    """float8_e4m3fn codes -> float64 values (same shape)."""
    a = _u8(codes)
    out = np.zeros(a.shape, dtype=np.float64)
    _check(_load().oracle_e4m3_decode(_ptr(a), _ptr(out), int(a.size)))
    return torch.from_numpy(out)


def attn_paged_fp8kv(q, k_cache, v_cache, k_scale, v_scale, real_seqlen_kv, block_table, causal=True,
                     scale=None, requests=None, nthreads=0, window_left=-1, window_right=-1, softcap=0.0,
                     sinks=None):
    """Paged GQA attention over float8_e4m3fn key/value caches, in double.

    q: [B,Sq,Hq,D] (16-bit or float); k_cache, v_cache: [num_pages, page_size,
    Hkv, D] e4m3fn codes (torch.float8_e4m3fn or uint8); k_scale, v_scale:
    [B, Hkv] dequantization scales (None: ones).  Key j of KV head r in
    request b is K * k_scale[b, r], its value V * v_scale[b, r] (TileOPs
    GQADenseFwdOp, FP8 dequantization).  Other arguments as attn_paged."""
    B, Sq, Hq, D = q.shape
    num_pages, page_size, Hkv, _ = k_cache.shape
    if scale is None:
        scale = default_scale(D)
    qa, c = _tensor_in(q)
    ka, va = _u8(k_cache), _u8(v_cache)

    def sc(x):
        if x is None:
            return None
        a = np.ascontiguousarray(torch.as_tensor(x).detach().cpu().to(torch.float64).numpy().reshape(-1))
        if a.shape[0] != B * Hkv:
            raise ValueError("oracle: k_scale / v_scale must hold one value per request and KV head")
        return a
    ks, vs = sc(k_scale), sc(v_scale)
    sl = np.ascontiguousarray(torch.as_tensor(real_seqlen_kv).cpu().numpy(), dtype=np.int32)
    bt = np.ascontiguousarray(torch.as_tensor(block_table).cpu().numpy(), dtype=np.int32)
    max_pages = bt.shape[1] if bt.ndim == 2 else 0
    req = None
    if requests is not None:
        req = np.zeros((B,), dtype=np.uint8)
        req[np.asarray(list(requests), dtype=np.int64)] = 1
    o = np.zeros((B, Sq, Hq, D), dtype=np.float64)
    lse = np.zeros((B, Sq, Hq), dtype=np.float64)
    wl, wr, cap, sk = _opts(window_left, window_right, softcap, sinks, Hq)
    rc = _load().oracle_attn_paged_fp8kv_ex(_ptr(qa), c, _ptr(ka), _ptr(va), _ptr(ks), _ptr(vs), _ptr(sl),
                                            _ptr(bt), page_size, _ptr(req), _ptr(o), _ptr(lse), B, Sq, Hq, Hkv,
                                            D, num_pages, max_pages, int(bool(causal)), float(scale), wl, wr,
                                            cap, _ptr(sk), int(nthreads))
    _check(rc)
    return torch.from_numpy(o), torch.from_numpy(lse)
