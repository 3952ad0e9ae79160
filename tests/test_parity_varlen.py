"""Packed variable-length calls on the GPU against the FP64 oracle, through
the C ABI: attn_fwd_varlen (TileOPs "Attention Operators", GQAVarlenFwdOp)
and attn_fwd_paged (GQAPagedFwdOp: prefill chunks and decode steps over a
paged cache in one launch).  Request mixes with empty requests, requests
without keys, Sq > Skv, group sizes that do not divide the 128-row tile,
every head dim, page sizes from 1 to 256, the optional terms, float16, and
cache slots the call must not read poisoned with NaN."""
import pytest
import torch

import oracle
from gqa_softmax_attention_gb300 import workloads as W

from parity import compare

pytestmark = pytest.mark.gpu

INF = float("inf")


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gqa_softmax_attention_gb300 import build
    build.build()
    import gqa_softmax_attention_gb300 as m
    yield m
    m.gqa_device_error()          # no kernel wait may have timed out


def check(o, lse, ro, rl, label):
    """compare(), with rows of a +inf sink (zero output, LSE +inf) checked apart."""
    o, lse = o.cpu(), lse.cpu()
    pos = torch.isposinf(rl)
    if bool(pos.any()):
        assert bool(torch.all(torch.isposinf(lse[pos]))) and bool(torch.all(o.float()[pos] == 0)), label
        o, lse, ro, rl = o[~pos], lse[~pos], ro[~pos], rl[~pos]
    return compare(o, lse, ro, rl, label)


def poison(p):
    """NaN into every cache slot no request may read: unused pages and the
    slots of a request's last page past its length."""
    kc, vc, table, L = p["k_cache"].clone(), p["v_cache"].clone(), p["block_table"], p["cache_seqlens"]
    ps = kc.shape[1]
    used = torch.zeros(kc.shape[0], dtype=torch.bool)
    for b in range(table.shape[0]):
        n = (int(L[b]) + ps - 1) // ps
        used[table[b, :n].long()] = True
        if n > 0 and int(L[b]) % ps:
            last = int(table[b, n - 1])
            kc[last, int(L[b]) % ps:] = float("nan")
            vc[last, int(L[b]) % ps:] = float("nan")
    kc[~used] = float("nan")
    vc[~used] = float("nan")
    return kc, vc


def sinks_for(Hq, seed):
    gen = torch.Generator().manual_seed(seed)
    s = torch.randn(Hq, generator=gen) * 2.0
    s[0], s[-1] = -INF, INF
    return s


VARLEN = [
    # q lengths, kv lengths, Hq, Hkv, D, causal
    ([1, 0, 200, 37, 129], [300, 5, 200, 37, 1000], 8, 2, 128, True),     # decode row, empty, prefill, chunk
    ([50, 3, 128], [20, 0, 500], 4, 4, 64, True),                          # Sq > Skv, no keys, MHA (g = 1)
    ([130, 1, 7, 64], [130, 900, 300, 64], 24, 2, 256, True),              # g = 12: 10 queries per block
    ([90, 250], [400, 250], 6, 2, 128, False),                             # non-causal
]


@pytest.mark.parametrize("case", VARLEN, ids=[str(c[:2]) for c in VARLEN])
def test_varlen(g, case):
    ql, kl, Hq, Hkv, D, causal = case
    d = W.varlen_inputs(ql, kl, Hq, Hkv, D, seed=sum(ql))
    dev = [d[n].cuda() for n in ("q", "k", "v", "cu_seqlens_q", "cu_seqlens_kv")]
    o, lse = g.varlen(*dev, causal=causal)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_varlen(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_kv"], causal=causal)
    check(o, lse, ro, rl, str(case))


def test_varlen_options_float16(g):
    ql, kl, Hq, Hkv, D = [70, 1, 260], [300, 40, 260], 8, 2, 128
    d = W.varlen_inputs(ql, kl, Hq, Hkv, D, seed=7)
    sinks = sinks_for(Hq, 3)
    for dtype in (torch.bfloat16, torch.float16):
        q, k, v = (d[n].to(dtype) for n in ("q", "k", "v"))
        kw = dict(window_left=100, window_right=-1, softcap=15.0, sinks=sinks)
        o, lse = g.varlen(q.cuda(), k.cuda(), v.cuda(), d["cu_seqlens_q"].cuda(), d["cu_seqlens_kv"].cuda(),
                          causal=True, **dict(kw, sinks=sinks.cuda()))
        torch.cuda.synchronize()
        assert o.dtype == dtype
        ro, rl = oracle.attn_varlen(q, k, v, d["cu_seqlens_q"], d["cu_seqlens_kv"], causal=True, **kw)
        check(o, lse, ro, rl, "options " + str(dtype))


PAGED = [
    # q lengths, cache lengths (query tokens included), Hq, Hkv, D, page_size
    ([1, 300, 0, 4, 1, 129], [1000, 800, 50, 333, 1, 129], 8, 2, 128, 16),
    ([1, 1, 1, 1, 2, 200], [17, 4000, 129, 640, 2, 200], 32, 8, 128, 64),
    ([4, 4, 1, 64], [3000, 17, 700, 64], 24, 2, 256, 16),                  # g = 12, D = 256
    ([3, 100, 1], [77, 100, 1000], 4, 2, 64, 8),
    ([1, 40, 2], [500, 300, 2], 8, 2, 128, 24),                            # 24-token pages: 8-token blocks
    ([5, 1, 130], [900, 600, 130], 16, 2, 256, 256),                       # pages larger than a key tile
    ([1, 1, 20, 1], [0, 700, 40, 1], 8, 2, 128, 16),                       # a decode step with an empty cache
    # page sizes that are not a multiple of 8: rows gathered with cp.async
    ([1, 37, 3], [300, 200, 3], 8, 2, 128, 1),
    ([2, 1, 150], [41, 500, 400], 8, 2, 64, 3),
    ([1, 129, 4], [777, 129, 260], 24, 2, 256, 5),
    ([200, 1, 1], [1000, 13, 1200], 32, 8, 128, 12),
]


@pytest.mark.parametrize("split_decode", [True, False], ids=["split_decode", "packed_only"])
@pytest.mark.parametrize("case", PAGED, ids=[str(c[:2]) + "/ps%d" % c[5] for c in PAGED])
def test_paged(g, case, split_decode):
    """With the larger workspace the one-query requests run on the split decode
    kernel and the rest on the packed kernel; with the packed workspace every
    request runs on the packed kernel.  Both against the oracle."""
    ql, L, Hq, Hkv, D, ps = case
    p = W.varlen_paged_inputs(ql, L, Hq, Hkv, D, ps, seed=sum(L) % 97)
    kc, vc = poison(p)
    o, lse = g.paged(p["q"].cuda(), kc.cuda(), vc.cuda(), p["cu_seqlens_q"].cuda(), p["cache_seqlens"].cuda(),
                     p["block_table"].cuda(), causal=True, split_decode=split_decode)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_paged_varlen(p["q"], p["k_cache"], p["v_cache"], p["cu_seqlens_q"], p["cache_seqlens"],
                                      p["block_table"], causal=True)
    check(o, lse, ro, rl, str(case))


@pytest.mark.parametrize("split_decode", [True, False], ids=["split_decode", "packed_only"])
def test_paged_options_float16(g, split_decode):
    ql, L, Hq, Hkv, D, ps = [1, 200, 4, 1], [2000, 450, 40, 90], 24, 2, 256, 32
    p = W.varlen_paged_inputs(ql, L, Hq, Hkv, D, ps, seed=5)
    sinks = sinks_for(Hq, 9)
    for dtype in (torch.bfloat16, torch.float16):
        q, kc, vc = (p[n].to(dtype) for n in ("q", "k_cache", "v_cache"))
        kw = dict(window_left=300, softcap=20.0)
        o, lse = g.paged(q.cuda(), kc.cuda(), vc.cuda(), p["cu_seqlens_q"].cuda(), p["cache_seqlens"].cuda(),
                         p["block_table"].cuda(), causal=True, sinks=sinks.cuda(), split_decode=split_decode, **kw)
        torch.cuda.synchronize()
        assert o.dtype == dtype
        ro, rl = oracle.attn_paged_varlen(q, kc, vc, p["cu_seqlens_q"], p["cache_seqlens"], p["block_table"],
                                          causal=True, sinks=sinks, **kw)
        check(o, lse, ro, rl, "paged options " + str(dtype))


def test_paged_decode_heavy_split(g):
    """Decode steps over long caches beside one short chunk: the plan leaves
    the chunk the fewest CTAs (the rest of the SMs go to the split decode
    kernel, which runs beside it on the caller's stream), and both parts match
    the oracle.  Then a chunk with no decode step keeps every CTA."""
    for ql, L in (([1] * 40 + [300], [6000 + 37 * i for i in range(40)] + [500]), ([300, 700], [500, 900])):
        Hq, Hkv, D, ps = 32, 8, 128, 64
        p = W.varlen_paged_inputs(ql, L, Hq, Hkv, D, ps, seed=len(ql))
        kc, vc = poison(p)
        tq = p["q"].shape[0]
        ws = torch.zeros(g.attn_paged_workspace_size(len(ql), tq, Hq, Hkv, D, ps, p["block_table"].shape[1]),
                         dtype=torch.uint8, device="cuda")
        o, lse = g.paged(p["q"].cuda(), kc.cuda(), vc.cuda(), p["cu_seqlens_q"].cuda(), p["cache_seqlens"].cuda(),
                         p["block_table"].cuda(), causal=True, workspace=ws)
        torch.cuda.synchronize()
        ro, rl = oracle.attn_paged_varlen(p["q"], p["k_cache"], p["v_cache"], p["cu_seqlens_q"], p["cache_seqlens"],
                                          p["block_table"], causal=True)
        check(o, lse, ro, rl, "decode-heavy split %d requests" % len(ql))
        # the plan's share of the persistent CTAs (third word of the workspace header)
        share = int(ws[:16].view(torch.int32)[2])
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        if ql[0] == 1:
            assert 8 <= share < sms // 4, share
        else:
            assert share == sms, share


def test_paged_equals_uniform_decode(g):
    """One query per request through the packed call equals the [B, 1] decode
    entry point (different kernels, same definition)."""
    p = W.paged_inputs(16, 1, 32, 8, 128, 64, lengths=(100, 3000), seed=2)
    cu = torch.arange(0, 17, dtype=torch.int32)
    o1, l1 = g.paged(p["q"][:, 0].cuda(), p["k_cache"].cuda(), p["v_cache"].cuda(), cu.cuda(),
                     p["real_seqlen_kv"].cuda(), p["block_table"].cuda(), causal=True)
    o2, l2 = g.decode_paged(p["q"].cuda(), p["k_cache"].cuda(), p["v_cache"].cuda(), p["real_seqlen_kv"].cuda(),
                            p["block_table"].cuda(), causal=True)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_paged(p["q"], p["k_cache"], p["v_cache"], p["real_seqlen_kv"], p["block_table"], causal=True)
    compare(o1.cpu(), l1.cpu(), ro[:, 0], rl[:, 0], "packed decode")
    compare(o2[:, 0].cpu(), l2[:, 0].cpu(), ro[:, 0], rl[:, 0], "decode")


def test_mixed_serving_batch_sampled(g):
    """A serving-sized mixed batch (two 2048-token prefill chunks over long
    caches and 62 decode steps, Qwen3-8B geometry): every request checked
    against the oracle on a sample of requests."""
    gen = torch.Generator().manual_seed(4)
    L = [int(x) for x in torch.randint(1024, 16385, (64,), generator=gen)]
    ql = [1] * 64
    ql[5], ql[40] = 2048, 2048
    L[5], L[40] = max(L[5], 4096), max(L[40], 2048)
    p = W.varlen_paged_inputs(ql, L, 32, 8, 128, 64, seed=11)
    kc, vc = poison(p)
    o, lse = g.paged(p["q"].cuda(), kc.cuda(), vc.cuda(), p["cu_seqlens_q"].cuda(), p["cache_seqlens"].cuda(),
                     p["block_table"].cuda(), causal=True)
    torch.cuda.synchronize()
    o, lse = o.cpu(), lse.cpu()
    assert not torch.isnan(o.float()).any() and bool(torch.isfinite(lse).all())
    cq, Ls = p["cu_seqlens_q"], p["cache_seqlens"]
    one = torch.tensor([0, 1], dtype=torch.int32)
    for b in (0, 5, 17, 40, 63):
        qs, sq = int(cq[b]), int(cq[b + 1] - cq[b])
        for i in sorted({0, 1, 127, 128, sq // 2, sq - 1} & set(range(sq))):
            # query i of request b sits at key position i + L_b - Sq_b: a
            # one-query request whose cache ends right after that position
            Li = torch.tensor([i + int(Ls[b]) - sq + 1], dtype=torch.int32)
            ro, rl = oracle.attn_paged_varlen(p["q"][qs + i:qs + i + 1], p["k_cache"], p["v_cache"], one, Li,
                                              p["block_table"][b:b + 1], causal=True)
            compare(o[qs + i:qs + i + 1], lse[qs + i:qs + i + 1], ro, rl, "request %d row %d" % (b, i))


def test_many_requests_plan(g):
    """More requests than the plan kernel's 1024 threads (its scan runs in
    chunks) and a cache shorter than the query count (leading rows see no key)."""
    gen = torch.Generator().manual_seed(21)
    B = 1500
    ql = torch.randint(0, 3, (B,), generator=gen).tolist()
    L = [max(1, int(x)) for x in torch.randint(1, 200, (B,), generator=gen)]
    L[7], ql[7] = 2, 3                                   # Sq > L: the first query sees nothing
    p = W.varlen_paged_inputs(ql, L, 4, 2, 64, 8, seed=3)
    o, lse = g.paged(p["q"].cuda(), p["k_cache"].cuda(), p["v_cache"].cuda(), p["cu_seqlens_q"].cuda(),
                     p["cache_seqlens"].cuda(), p["block_table"].cuda(), causal=True)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_paged_varlen(p["q"], p["k_cache"], p["v_cache"], p["cu_seqlens_q"], p["cache_seqlens"],
                                      p["block_table"], causal=True)
    compare(o.cpu(), lse.cpu(), ro, rl, "1500 requests")
    qs = int(p["cu_seqlens_q"][7])
    assert bool(torch.isneginf(lse[qs, :].cpu()).all())


def test_varlen_two_sided_window_noncausal(g):
    ql, kl, Hq, Hkv, D = [60, 200, 5], [300, 200, 90], 6, 3, 128
    d = W.varlen_inputs(ql, kl, Hq, Hkv, D, seed=12)
    o, lse = g.varlen(*[d[n].cuda() for n in ("q", "k", "v", "cu_seqlens_q", "cu_seqlens_kv")], causal=False,
                      window_left=40, window_right=17)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_varlen(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_kv"], causal=False,
                                window_left=40, window_right=17)
    compare(o.cpu(), lse.cpu(), ro, rl, "two-sided window")
