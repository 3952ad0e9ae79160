"""Python entry points with the C ABI's names; torch supplies memory and streams.

Every step of the computation runs in libgqa_attn.so.  These functions check
dtypes and devices, make inputs contiguous (TileOPs GQADenseFwdOp, forward:
non-contiguous inputs are copied first), resolve ``scale=None`` to 1/sqrt(D)
(RL-Kernel Tensor Contract), allocate outputs with torch and pass raw pointers
plus the current CUDA stream.  A non-OK status raises: ``ValueError`` for
argument problems (naming the refused limit), ``RuntimeError`` for CUDA errors.
"""
import ctypes
import math

import torch

from . import _lib

_ARG_ERRORS = {1, 2, 3, 4}


def _raise(status: int, what: str):
    name = _lib.status_name(status)
    msg = "%s: %s (%s)" % (what, _lib.load().gqa_status_string(status).decode(), name)
    if status in _ARG_ERRORS:
        raise ValueError(msg)
    raise RuntimeError(msg)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


_DTYPES = {torch.bfloat16: 0, torch.float16: 1}      # gqa_dtype


def _check_16_cuda(name, t, ndim, dtypes=(torch.bfloat16, torch.float16)):
    """A CUDA tensor of ndim dimensions and one of the given dtypes."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype not in dtypes:
        raise ValueError("%s must be %s, got %s" % (name, " or ".join(str(d) for d in dtypes), t.dtype))
    if t.dim() != ndim:
        raise ValueError("%s must have %d dimensions, got %d" % (name, ndim, t.dim()))


def resolve_scale(scale, D):
    """None -> 1/sqrt(D); an explicit value (0.0 included) is used verbatim."""
    return 1.0 / math.sqrt(D) if scale is None else float(scale)


def _options(window_left, window_right, softcap, sinks, Hq, device, dtype=0):
    """gqa_options for the optional terms and the element type, or None when
    none is set (the sinks tensor is returned too, to keep it alive for the
    call)."""
    if window_left == -1 and window_right == -1 and not softcap and sinks is None and dtype == 0:
        return None, None
    for n, w in (("window_left", window_left), ("window_right", window_right)):
        if int(w) < -1:
            raise ValueError("%s must be -1 (unlimited) or >= 0, got %d" % (n, int(w)))
    cap = 0.0 if softcap is None else float(softcap)
    if not math.isfinite(cap) or cap < 0.0:
        raise ValueError("softcap must be finite and >= 0, got %r" % (softcap,))
    sk = None
    if sinks is not None:
        sk = torch.as_tensor(sinks).to(device=device, dtype=torch.float32).contiguous()
        if tuple(sk.shape) != (Hq,):
            raise ValueError("sinks must be [Hq] = [%d]" % Hq)
    opt = _lib.Options(int(window_left), int(window_right), cap, sk.data_ptr() if sk is not None else None,
                       int(dtype))
    return opt, sk


def attn_fwd_dense(q, k, v, key_padding_mask=None, causal=True, scale=None, out=None, lse=None,
                   window_left=-1, window_right=-1, softcap=None, sinks=None):
    """Dense / chunked-prefill GQA attention.

    q [B,Sq,Hq,D], k/v [B,Skv,Hkv,D] CUDA tensors (BSHD), all bfloat16 or all
    float16 (the output takes the same type);
    key_padding_mask [B,Skv] bool (True = keep) or None.
    window_left / window_right: keys admitted left / right of each query's key
    position (-1 unlimited); softcap: c > 0 caps each scaled score to
    c*tanh(z/c) (None or 0 off); sinks: [Hq] float32 logits joining the
    softmax denominator only, or None.
    Returns (o [B,Sq,Hq,D] bf16, lse [B,Sq,Hq] float32, natural log).
    """
    _check_16_cuda("q", q, 4)
    for n, t in (("k", k), ("v", v)):
        _check_16_cuda(n, t, 4, (q.dtype,))
    B, Sq, Hq, D = q.shape
    Bk, Skv, Hkv, Dk = k.shape
    if Bk != B or Dk != D or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch: q %s, k %s, v %s" % (tuple(q.shape), tuple(k.shape), tuple(v.shape)))
    if Hq % Hkv != 0:
        raise ValueError("Hq (%d) must be divisible by Hkv (%d)" % (Hq, Hkv))
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    m = None
    if key_padding_mask is not None:
        if tuple(key_padding_mask.shape) != (B, Skv):
            raise ValueError("key_padding_mask must be [B, Skv] = [%d, %d]" % (B, Skv))
        m = key_padding_mask.to(device=q.device, dtype=torch.bool).contiguous().view(torch.uint8)
    if out is None:
        out = torch.empty((B, Sq, Hq, D), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Sq, Hq), dtype=torch.float32, device=q.device)
    opt, _keep = _options(window_left, window_right, softcap, sinks, Hq, q.device, _DTYPES[q.dtype])
    lib = _lib.load()
    if opt is None:
        st = lib.attn_fwd_dense(_ptr(q), _ptr(k), _ptr(v), _ptr(m), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Skv, D,
                                int(bool(causal)), resolve_scale(scale, D), _stream(q.device))
    else:
        st = lib.attn_fwd_dense_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(m), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Skv,
                                   D, int(bool(causal)), resolve_scale(scale, D), ctypes.byref(opt),
                                   _stream(q.device))
    if st != 0:
        _raise(st, "attn_fwd_dense")
    return out, lse


def _check_paged(q, k_cache, v_cache, real_seqlen_kv, block_table, dtypes=(torch.bfloat16, torch.float16)):
    """Checks shared by the paged decode entry points: q [B,Sq,Hq,D] and the
    caches [num_pages,page_size,Hkv,D] CUDA tensors of one 16-bit type, Hq a
    multiple of Hkv, real_seqlen_kv [B] and block_table [B,max_pages] int32 CUDA
    tensors.  Returns the five tensors made contiguous."""
    _check_16_cuda("q", q, 4, dtypes)
    _check_16_cuda("k_cache", k_cache, 4, (q.dtype,))
    _check_16_cuda("v_cache", v_cache, 4, (q.dtype,))
    B, Sq, Hq, D = q.shape
    num_pages, page_size, Hkv, Dk = k_cache.shape
    if Dk != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shape mismatch: k %s, v %s, D %d" % (tuple(k_cache.shape), tuple(v_cache.shape), D))
    if Hq % Hkv != 0:
        raise ValueError("Hq (%d) must be divisible by Hkv (%d)" % (Hq, Hkv))
    for n, t in (("real_seqlen_kv", real_seqlen_kv), ("block_table", block_table)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.int32:
            raise ValueError("%s must be an int32 CUDA tensor" % n)
        if t.device != q.device:
            raise ValueError("%s must be on q's device %s, got %s" % (n, q.device, t.device))
    if tuple(real_seqlen_kv.shape) != (B,) or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("real_seqlen_kv must be [B] and block_table [B, max_pages]")
    return (q.contiguous(), k_cache.contiguous(), v_cache.contiguous(), real_seqlen_kv.contiguous(),
            block_table.contiguous())


def attn_decode_paged_workspace_size(B, Sq, Hq, Hkv, D, page_size, max_pages):
    """Workspace bytes attn_decode_paged needs on the current device."""
    return int(_lib.load().attn_decode_paged_workspace_size(B, Sq, Hq, Hkv, D, page_size, max_pages))


def attn_decode_paged(q, k_cache, v_cache, real_seqlen_kv, block_table, causal=True, scale=None,
                      workspace=None, out=None, lse=None, window_left=-1, window_right=-1, softcap=None,
                      sinks=None):
    """Paged decode.

    q [B,Sq,Hq,D]; k_cache/v_cache [num_pages,page_size,Hkv,D], all bfloat16 or all float16;
    real_seqlen_kv [B] int32 (query tokens included); block_table [B,max_pages] int32.
    workspace: optional uint8 CUDA tensor of at least attn_decode_paged_workspace_size bytes.
    window_left / window_right / softcap / sinks as in attn_fwd_dense.
    Returns (o [B,Sq,Hq,D] bf16, lse [B,Sq,Hq] float32).
    """
    q, k_cache, v_cache, sl, bt = _check_paged(q, k_cache, v_cache, real_seqlen_kv, block_table)
    B, Sq, Hq, D = q.shape
    num_pages, page_size, Hkv, _ = k_cache.shape
    max_pages = bt.shape[1]
    need = attn_decode_paged_workspace_size(B, Sq, Hq, Hkv, D, page_size, max_pages)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty((B, Sq, Hq, D), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Sq, Hq), dtype=torch.float32, device=q.device)
    opt, _keep = _options(window_left, window_right, softcap, sinks, Hq, q.device, _DTYPES[q.dtype])
    lib = _lib.load()
    wsb = workspace.numel() * workspace.element_size()
    if opt is None:
        st = lib.attn_decode_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(sl), _ptr(bt), page_size,
                                   _ptr(out), _ptr(lse), B, Sq, Hq, Hkv, D, num_pages, max_pages,
                                   int(bool(causal)), resolve_scale(scale, D), _ptr(workspace), wsb,
                                   _stream(q.device))
    else:
        st = lib.attn_decode_paged_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(sl), _ptr(bt), page_size,
                                      _ptr(out), _ptr(lse), B, Sq, Hq, Hkv, D, num_pages, max_pages,
                                      int(bool(causal)), resolve_scale(scale, D), ctypes.byref(opt),
                                      _ptr(workspace), wsb, _stream(q.device))
    if st != 0:
        _raise(st, "attn_decode_paged")
    return out, lse


def attn_decode_paged_fp8kv(q, k_cache, v_cache, k_scale, v_scale, real_seqlen_kv, block_table, causal=True,
                            scale=None, workspace=None, out=None, lse=None, window_left=-1, window_right=-1,
                            softcap=None, sinks=None):
    """Paged decode over float8_e4m3fn key/value caches.

    q [B,Sq,Hq,D] bfloat16 or float16; k_cache/v_cache [num_pages,page_size,Hkv,D]
    torch.float8_e4m3fn (or uint8 holding e4m3fn codes); k_scale/v_scale [B,Hkv]
    float32 CUDA tensors or None (ones): key t of KV head r in request b is
    K * k_scale[b, r] and its value V * v_scale[b, r].  Every scale must be finite
    and positive; they stay on the GPU and are not checked.  D is 128 or 256.  Other
    arguments as attn_decode_paged.  Returns (o like q, lse [B,Sq,Hq] float32).
    """
    _check_16_cuda("q", q, 4)
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dim() != 4 or \
                t.dtype not in (torch.float8_e4m3fn, torch.uint8):
            raise ValueError("%s must be a 4-D float8_e4m3fn (or uint8) CUDA tensor" % n)
    B, Sq, Hq, D = q.shape
    num_pages, page_size, Hkv, Dk = k_cache.shape
    if Dk != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shape mismatch: k %s, v %s, D %d" % (tuple(k_cache.shape), tuple(v_cache.shape), D))
    if Hq % Hkv != 0:
        raise ValueError("Hq (%d) must be divisible by Hkv (%d)" % (Hq, Hkv))
    for n, t in (("real_seqlen_kv", real_seqlen_kv), ("block_table", block_table)):
        if not t.is_cuda or t.dtype != torch.int32:
            raise ValueError("%s must be an int32 CUDA tensor" % n)
    if tuple(real_seqlen_kv.shape) != (B,) or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("real_seqlen_kv must be [B] and block_table [B, max_pages]")
    scales = []
    for n, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        if t is not None:
            if not t.is_cuda or t.dtype != torch.float32 or t.numel() != B * Hkv:
                raise ValueError("%s must be a float32 CUDA tensor of B * Hkv values" % n)
            t = t.contiguous()
        scales.append(t)
    max_pages = block_table.shape[1]
    q, k_cache, v_cache = q.contiguous(), k_cache.contiguous(), v_cache.contiguous()
    sl, bt = real_seqlen_kv.contiguous(), block_table.contiguous()
    need = attn_decode_paged_workspace_size(B, Sq, Hq, Hkv, D, page_size, max_pages)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty((B, Sq, Hq, D), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Sq, Hq), dtype=torch.float32, device=q.device)
    opt, _keep = _options(window_left, window_right, softcap, sinks, Hq, q.device, _DTYPES[q.dtype])
    st = _lib.load().attn_decode_paged_fp8kv(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(scales[0]), _ptr(scales[1]), _ptr(sl), _ptr(bt), page_size,
        _ptr(out), _ptr(lse), B, Sq, Hq, Hkv, D, num_pages, max_pages, int(bool(causal)), resolve_scale(scale, D),
        ctypes.byref(opt) if opt is not None else None, _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(q.device))
    if st != 0:
        _raise(st, "attn_decode_paged_fp8kv")
    return out, lse


def attn_decode_paged_noalloc(q, k_cache, v_cache, real_seqlen_kv, block_table, causal=True, scale=None, out=None,
                              lse=None):
    """Paged decode through the entry point that allocates nothing in the library.

    For callers that cannot allocate device memory or supply a workspace: the
    split partials go to a fixed 32 MiB array inside the library, shared by all
    calls (calls overlapping on the GPU race).  Sizes whose partials do not fit
    raise ValueError.  Outputs are allocated here only when not passed in.
    """
    q, k_cache, v_cache, real_seqlen_kv, block_table = _check_paged(q, k_cache, v_cache, real_seqlen_kv,
                                                                    block_table, (torch.bfloat16,))
    B, Sq, Hq, D = q.shape
    num_pages, page_size, Hkv, _ = k_cache.shape
    max_pages = block_table.shape[1]
    if out is None:
        out = torch.empty((B, Sq, Hq, D), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, Sq, Hq), dtype=torch.float32, device=q.device)
    st = _lib.load().attn_decode_paged_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(real_seqlen_kv),
                                               _ptr(block_table), page_size, _ptr(out), _ptr(lse), B, Sq, Hq, Hkv,
                                               D, num_pages, max_pages, int(bool(causal)),
                                               resolve_scale(scale, D), _stream(q.device))
    if st != 0:
        _raise(st, "attn_decode_paged_noalloc (static scratch %d bytes)"
               % _lib.load().attn_decode_paged_noalloc_max_workspace())
    return out, lse


def attn_varlen_workspace_size(B, total_q, Hq, Hkv):
    """Workspace bytes of attn_fwd_varlen / attn_fwd_paged."""
    return int(_lib.load().attn_varlen_workspace_size(B, total_q, Hq, Hkv))


def attn_paged_workspace_size(B, total_q, Hq, Hkv, D, page_size, max_pages):
    """Workspace bytes of attn_fwd_paged with its single-query requests on the
    split-KV decode kernel (equal to attn_varlen_workspace_size when the sizes
    keep every request on the packed kernel)."""
    return int(_lib.load().attn_paged_workspace_size(B, total_q, Hq, Hkv, D, page_size, max_pages))


def _check_offsets(name, t, n):
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.int32 or tuple(t.shape) != (n,):
        raise ValueError("%s must be an int32 CUDA tensor of shape [%d]" % (name, n))
    return t.contiguous()


def _varlen_outputs(q, out, lse, workspace, B):
    total_q, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    return out, lse


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_kv, causal=True, scale=None, out=None, lse=None,
                    window_left=-1, window_right=-1, softcap=None, sinks=None, workspace=None):
    """Packed variable-length GQA attention (TileOPs GQAVarlenFwdOp).

    q [total_q, Hq, D], k / v [total_kv, Hkv, D] CUDA tensors (THD), all
    bfloat16 or all float16; cu_seqlens_q / cu_seqlens_kv [B + 1] int32 CUDA
    offsets (request b owns rows cu[b]:cu[b+1]; they stay on the device).
    Options as in attn_fwd_dense.  Returns (o [total_q, Hq, D], lse [total_q, Hq]).
    """
    _check_16_cuda("q", q, 3)
    for n, t in (("k", k), ("v", v)):
        _check_16_cuda(n, t, 3, (q.dtype,))
    total_q, Hq, D = q.shape
    total_kv, Hkv, Dk = k.shape
    if Dk != D or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch: q %s, k %s, v %s" % (tuple(q.shape), tuple(k.shape), tuple(v.shape)))
    if Hq % Hkv != 0:
        raise ValueError("Hq (%d) must be divisible by Hkv (%d)" % (Hq, Hkv))
    if cu_seqlens_q.dim() != 1 or cu_seqlens_q.shape[0] < 2:
        raise ValueError("cu_seqlens_q must hold B + 1 >= 2 offsets")
    B = cu_seqlens_q.shape[0] - 1
    cq = _check_offsets("cu_seqlens_q", cu_seqlens_q, B + 1)
    ck = _check_offsets("cu_seqlens_kv", cu_seqlens_kv, B + 1)
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    out, lse = _varlen_outputs(q, out, lse, workspace, B)
    need = attn_varlen_workspace_size(B, total_q, Hq, Hkv)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    opt, _keep = _options(window_left, window_right, softcap, sinks, Hq, q.device, _DTYPES[q.dtype])
    st = _lib.load().attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(cq), _ptr(ck), _ptr(out), _ptr(lse), B, total_q,
                                     total_kv, Hq, Hkv, D, int(bool(causal)), resolve_scale(scale, D),
                                     ctypes.byref(opt) if opt is not None else None, _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(q.device))
    if st != 0:
        _raise(st, "attn_fwd_varlen")
    return out, lse


def attn_fwd_paged(q, k_cache, v_cache, cu_seqlens_q, cache_seqlens, block_table, causal=True, scale=None,
                   out=None, lse=None, window_left=-1, window_right=-1, softcap=None, sinks=None, workspace=None,
                   split_decode=True):
    """Packed queries over a paged cache: prefill chunks and decode steps in one
    call (TileOPs GQAPagedFwdOp).

    q [total_q, Hq, D]; k_cache / v_cache [num_pages, page_size, Hkv, D], all
    bfloat16 or all float16; cu_seqlens_q [B + 1], cache_seqlens [B] (query
    tokens included) and block_table [B, max_pages] int32 CUDA tensors.
    Any page size (multiples of 8 move by TMA, others are gathered row by
    row).  Options as in attn_fwd_dense.
    split_decode: give the call the workspace that sends requests with one
    query to the split-KV decode kernel (False: every request on the packed
    kernel).  A caller's workspace decides by its size instead.  With the
    split, the packed kernel runs beside the decode kernel on a library-owned
    high-priority stream, forked from and joined back into the current stream
    inside the call.
    Returns (o [total_q, Hq, D], lse [total_q, Hq]).
    """
    _check_16_cuda("q", q, 3)
    _check_16_cuda("k_cache", k_cache, 4, (q.dtype,))
    _check_16_cuda("v_cache", v_cache, 4, (q.dtype,))
    total_q, Hq, D = q.shape
    num_pages, page_size, Hkv, Dk = k_cache.shape
    if Dk != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shape mismatch: k %s, v %s, D %d" % (tuple(k_cache.shape), tuple(v_cache.shape), D))
    if Hq % Hkv != 0:
        raise ValueError("Hq (%d) must be divisible by Hkv (%d)" % (Hq, Hkv))
    if cache_seqlens.dim() != 1:
        raise ValueError("cache_seqlens must be [B]")
    B = cache_seqlens.shape[0]
    cq = _check_offsets("cu_seqlens_q", cu_seqlens_q, B + 1)
    sl = _check_offsets("cache_seqlens", cache_seqlens, B)
    if not block_table.is_cuda or block_table.dtype != torch.int32 or block_table.dim() != 2 \
            or block_table.shape[0] != B:
        raise ValueError("block_table must be an int32 CUDA tensor [B, max_pages]")
    bt = block_table.contiguous()
    q, k_cache, v_cache = q.contiguous(), k_cache.contiguous(), v_cache.contiguous()
    out, lse = _varlen_outputs(q, out, lse, workspace, B)
    if split_decode:
        need = attn_paged_workspace_size(B, total_q, Hq, Hkv, D, page_size, bt.shape[1])
    else:
        need = attn_varlen_workspace_size(B, total_q, Hq, Hkv)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    opt, _keep = _options(window_left, window_right, softcap, sinks, Hq, q.device, _DTYPES[q.dtype])
    st = _lib.load().attn_fwd_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cq), _ptr(sl), _ptr(bt), page_size,
                                    _ptr(out), _ptr(lse), B, total_q, Hq, Hkv, D, num_pages, bt.shape[1],
                                    int(bool(causal)), resolve_scale(scale, D),
                                    ctypes.byref(opt) if opt is not None else None, _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(q.device))
    if st != 0:
        _raise(st, "attn_fwd_paged")
    return out, lse


def attn_validate_paged(real_seqlen_kv, block_table, Sq, page_size, num_pages, causal=True):
    """Host-side range check of paged metadata (synchronises the stream)."""
    B, max_pages = block_table.shape
    st = _lib.load().attn_validate_paged(_ptr(real_seqlen_kv.contiguous()), _ptr(block_table.contiguous()), B, Sq,
                                         page_size, num_pages, max_pages, int(bool(causal)),
                                         _stream(block_table.device))
    if st != 0:
        _raise(st, "attn_validate_paged")


def gqa_device_error():
    """Raise if a kernel recorded a timed-out wait since the last check (synchronises)."""
    st = _lib.load().gqa_device_error()
    if st != 0:
        _raise(st, "gqa_device_error")


# Short aliases in the style of the pages' op APIs.
attention = attn_fwd_dense
decode_paged = attn_decode_paged
varlen = attn_fwd_varlen
paged = attn_fwd_paged
