"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random tensors and lays them out; it holds none of the
attention arithmetic and imports neither the CUDA binding nor the oracle, so
both sides consume exactly the same bytes.

Recipe (every draw on the CPU, float32 N(0, sigma^2) rounded to bfloat16 with
round-to-nearest-even):

* A tensor is drawn as a flat sequence cut into chunks of ``CHUNK`` elements;
  chunk c of stream s comes from ``torch.Generator().manual_seed(
  seed * 2**32 + s * 2**20 + c)``.  Chunks are independent, so large pools are
  drawn on several host threads with an unchanged result.
* Dense: streams 0, 1, 2 are q, k, v.  With a padding mask, the per-batch valid
  lengths come from ``torch.randint(lo, hi + 1, (B,))`` on
  ``Generator().manual_seed(seed)`` and ``mask[b, j] = j < L_b``.
* Paged: the lengths L_b are drawn first on ``Generator().manual_seed(seed)``
  (the pool size depends on them), then the page permutation
  ``torch.randperm(pool)`` on the same generator.  The pool holds
  ``sum_b ceil(L_b / page_size)`` used pages plus ``ceil(spare * used)`` unused
  ones; request b's logical pages take the next ``ceil(L_b / page_size)``
  entries of the permutation, in request order; unused block_table entries are
  -1.  Streams 0, 1, 2 are q, k_cache, v_cache.
* Paged FP8: the paged draw, each bf16 cache value rounded to float8_e4m3fn
  by torch, then ``k_scale`` and ``v_scale`` [B, Hkv] uniform on the workload's
  scale range from ``Generator().manual_seed(seed * 2**32 + 3 * 2**20)``.

The named workloads are the shapes of the pages' examples: a tiny GQA case, a
Qwen3-8B-shaped prefill (Hq=32, Hkv=8, D=128), a paged decode batch of the same
geometry, a 24/2/D256 multi-query decode, a long chunked prefill, and a dense
causal prefill of the 24/2/D256 geometry.
"""
import math
from concurrent.futures import ThreadPoolExecutor

import torch

CHUNK = 1 << 22

WORKLOADS = {
    "tiny_dense": dict(kind="dense", B=1, Hq=4, Hkv=2, Sq=128, Skv=128, D=64, causal=True,
                       sigma=1.0, mask_lengths=None),
    "qwen3_8b_prefill": dict(kind="dense", B=2, Hq=32, Hkv=8, Sq=4096, Skv=4096, D=128,
                             causal=True, sigma=1.0, mask_lengths=(2048, 4096)),
    "paged_decode": dict(kind="paged", B=64, Sq=1, Hq=32, Hkv=8, D=128, page_size=64,
                         causal=True, sigma=1.0, lengths=(1024, 16384), spare=0.10),
    "wide_group_decode": dict(kind="paged", B=32, Sq=4, Hq=24, Hkv=2, D=256, page_size=16,
                              causal=True, sigma=1.0, lengths=(512, 32768), spare=0.10),
    "long_chunked_prefill": dict(kind="dense", B=4, Hq=64, Hkv=8, Sq=2048, Skv=32768, D=128,
                                 causal=True, sigma=0.5, mask_lengths=None),
    "wide_group_prefill": dict(kind="dense", B=2, Hq=24, Hkv=2, Sq=8192, Skv=8192, D=256,
                               causal=True, sigma=1.0, mask_lengths=None),
    # packed (THD) self-attention prefill of 16 requests of mixed length
    "varlen_prefill": dict(kind="varlen", B=16, Hq=32, Hkv=8, D=128, causal=True, sigma=1.0,
                           lengths=(256, 8192)),
    # the paged decode batch over float8_e4m3fn caches with per-(request, KV head) scales
    "paged_decode_fp8kv": dict(kind="paged_fp8", B=64, Sq=1, Hq=32, Hkv=8, D=128, page_size=64, causal=True,
                               sigma=1.0, lengths=(1024, 16384), spare=0.10, scale_range=(0.25, 1.0)),
    "wide_group_decode_fp8kv": dict(kind="paged_fp8", B=32, Sq=4, Hq=24, Hkv=2, D=256, page_size=16, causal=True,
                                    sigma=1.0, lengths=(512, 32768), spare=0.10, scale_range=(0.25, 1.0)),
    # one serving step over a paged cache: 60 decode steps (one query each,
    # cache lengths U[1024, 16384]) and 4 prefill chunks of 1024 queries whose
    # caches hold U[0, 8192] earlier tokens plus the chunk
    "mixed_serving_batch": dict(kind="paged_varlen", B=64, Hq=32, Hkv=8, D=128, page_size=64, causal=True,
                                sigma=1.0, decode_lengths=(1024, 16384), prefill_chunks=4, chunk=1024,
                                context=(0, 8192)),
}


def _draw_chunk(seed, stream, c, n, sigma):
    g = torch.Generator().manual_seed(seed * 2**32 + stream * 2**20 + c)
    x = torch.randn(n, generator=g, dtype=torch.float32)
    if sigma != 1.0:
        x.mul_(sigma)
    return x.to(torch.bfloat16)


def randn_bf16(shape, sigma=1.0, seed=0, stream=0, threads=None):
    """N(0, sigma^2) bfloat16 tensor of ``shape`` drawn by the chunked recipe."""
    numel = math.prod(shape)
    out = torch.empty(numel, dtype=torch.bfloat16)
    nchunks = (numel + CHUNK - 1) // CHUNK

    def work(c):
        lo = c * CHUNK
        hi = min(numel, lo + CHUNK)
        out[lo:hi] = _draw_chunk(seed, stream, c, hi - lo, sigma)

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(max_workers=threads or min(16, nchunks)) as ex:
            list(ex.map(work, range(nchunks)))
    return out.view(*shape)


def dense_inputs(B, Hq, Hkv, Sq, Skv, D, sigma=1.0, mask_lengths=None, seed=0, **_):
    """q [B,Sq,Hq,D], k/v [B,Skv,Hkv,D] bf16, optional key_padding_mask [B,Skv] bool."""
    q = randn_bf16((B, Sq, Hq, D), sigma, seed, 0)
    k = randn_bf16((B, Skv, Hkv, D), sigma, seed, 1)
    v = randn_bf16((B, Skv, Hkv, D), sigma, seed, 2)
    mask, lengths = None, None
    if mask_lengths is not None:
        lo, hi = mask_lengths
        g = torch.Generator().manual_seed(seed)
        lengths = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64)
        mask = torch.arange(Skv)[None, :] < lengths[:, None]
    return dict(q=q, k=k, v=v, key_padding_mask=mask, lengths=lengths)


def paged_inputs(B, Sq, Hq, Hkv, D, page_size, lengths, spare=0.10, sigma=1.0, seed=0,
                 max_pages=None, **_):
    """Paged decode inputs.

    lengths: a tuple (lo, hi) drawn uniformly, or a list / tensor of B lengths.
    Returns q [B,Sq,Hq,D], k_cache/v_cache [pool,page_size,Hkv,D] bf16,
    real_seqlen_kv [B] int32, block_table [B,max_pages] int32.
    """
    g = torch.Generator().manual_seed(seed)
    if isinstance(lengths, tuple):            # (lo, hi): uniform draw
        lo, hi = lengths
        L = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64)
        cap = hi
    else:                                     # explicit per-request lengths
        L = torch.as_tensor(list(lengths), dtype=torch.int64).reshape(B)
        cap = int(L.max()) if B > 0 else 0
    npages = (L + page_size - 1) // page_size
    used = int(npages.sum())
    pool = used + int(math.ceil(spare * used))
    if max_pages is None:
        max_pages = max(1, (cap + page_size - 1) // page_size)
    perm = torch.randperm(pool, generator=g).to(torch.int32) if pool > 0 else \
        torch.zeros(0, dtype=torch.int32)
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    off = 0
    for b in range(B):
        n = int(npages[b])
        table[b, :n] = perm[off:off + n]
        off += n
    q = randn_bf16((B, Sq, Hq, D), sigma, seed, 0)
    k_cache = randn_bf16((pool, page_size, Hkv, D), sigma, seed, 1)
    v_cache = randn_bf16((pool, page_size, Hkv, D), sigma, seed, 2)
    return dict(q=q, k_cache=k_cache, v_cache=v_cache, real_seqlen_kv=L.to(torch.int32),
                block_table=table, num_pages=pool, max_pages=max_pages, page_size=page_size)


def paged_fp8_inputs(B, Sq, Hq, Hkv, D, page_size, lengths, spare=0.10, sigma=1.0, seed=0,
                     scale_range=(0.25, 1.0), max_pages=None, **_):
    """Paged decode inputs with float8_e4m3fn caches: the paged_inputs draw,
    each bf16 cache value rounded to e4m3fn by torch (round to nearest even),
    and k_scale / v_scale [B, Hkv] float32 drawn uniformly from scale_range
    (stream 3, K first).  Returns the paged_inputs dict with k_cache / v_cache
    as torch.float8_e4m3fn and k_scale / v_scale added."""
    p = paged_inputs(B, Sq, Hq, Hkv, D, page_size, lengths, spare=spare, sigma=sigma, seed=seed,
                     max_pages=max_pages)
    p["k_cache"] = p["k_cache"].float().to(torch.float8_e4m3fn)
    p["v_cache"] = p["v_cache"].float().to(torch.float8_e4m3fn)
    g = torch.Generator().manual_seed(seed * 2**32 + 3 * 2**20)
    lo, hi = scale_range
    p["k_scale"] = lo + (hi - lo) * torch.rand(B, Hkv, generator=g, dtype=torch.float32)
    p["v_scale"] = lo + (hi - lo) * torch.rand(B, Hkv, generator=g, dtype=torch.float32)
    return p


def _offsets(lengths):
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def varlen_inputs(q_lens, kv_lens, Hq, Hkv, D, sigma=1.0, seed=0, **_):
    """Packed (THD) inputs: q [sum(q_lens), Hq, D], k / v [sum(kv_lens), Hkv, D]
    (streams 0, 1, 2) and their [B + 1] offsets."""
    cq, ck = _offsets(q_lens), _offsets(kv_lens)
    tq, tk = int(cq[-1]), int(ck[-1])
    q = randn_bf16((max(tq, 1), Hq, D), sigma, seed, 0)[:tq]
    k = randn_bf16((max(tk, 1), Hkv, D), sigma, seed, 1)[:tk]
    v = randn_bf16((max(tk, 1), Hkv, D), sigma, seed, 2)[:tk]
    return dict(q=q, k=k, v=v, cu_seqlens_q=cq, cu_seqlens_kv=ck)


def varlen_paged_inputs(q_lens, lengths, Hq, Hkv, D, page_size, spare=0.10, sigma=1.0, seed=0, **_):
    """Packed queries over a paged cache: the cache, lengths and table of
    paged_inputs(lengths) plus q [sum(q_lens), Hq, D] (stream 3) and its
    [B + 1] offsets; cache_seqlens = lengths (query tokens included)."""
    B = len(lengths)
    p = paged_inputs(B, 1, Hq, Hkv, D, page_size, list(lengths), spare=spare, sigma=sigma, seed=seed)
    cq = _offsets(q_lens)
    tq = int(cq[-1])
    p["q"] = randn_bf16((max(tq, 1), Hq, D), sigma, seed, 3)[:tq]
    p["cu_seqlens_q"] = cq
    p["cache_seqlens"] = p.pop("real_seqlen_kv")
    return p


def mixed_lengths(cfg, seed=0):
    """Per-request query counts and cache lengths of a paged_varlen workload:
    requests 0 .. chunks-1 are prefill chunks, the rest single decode steps
    (lengths on Generator().manual_seed(seed + 1))."""
    g = torch.Generator().manual_seed(seed + 1)
    B, nc, chunk = cfg["B"], cfg["prefill_chunks"], cfg["chunk"]
    lo, hi = cfg["decode_lengths"]
    clo, chi = cfg["context"]
    dec = torch.randint(lo, hi + 1, (B - nc,), generator=g).tolist()
    ctx = torch.randint(clo, chi + 1, (nc,), generator=g).tolist()
    q_lens = [chunk] * nc + [1] * (B - nc)
    lengths = [c + chunk for c in ctx] + dec
    return q_lens, lengths


def make(name, seed=0):
    """Inputs of a named workload plus its shape description."""
    cfg = dict(WORKLOADS[name])
    if cfg["kind"] == "dense":
        data = dense_inputs(seed=seed, **cfg)
    elif cfg["kind"] == "varlen":
        g = torch.Generator().manual_seed(seed + 1)
        lo, hi = cfg["lengths"]
        lens = torch.randint(lo, hi + 1, (cfg["B"],), generator=g).tolist()
        data = varlen_inputs(lens, lens, cfg["Hq"], cfg["Hkv"], cfg["D"], sigma=cfg["sigma"], seed=seed)
    elif cfg["kind"] == "paged_varlen":
        q_lens, lengths = mixed_lengths(cfg, seed)
        data = varlen_paged_inputs(q_lens, lengths, cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["page_size"],
                                   sigma=cfg["sigma"], seed=seed)
    elif cfg["kind"] == "paged_fp8":
        data = paged_fp8_inputs(seed=seed, **cfg)
    else:
        data = paged_inputs(seed=seed, **cfg)
    data["config"] = cfg
    return data
