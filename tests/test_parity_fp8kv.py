"""Paged decode over float8_e4m3fn key/value caches on the GPU against the FP64
oracle (through the C ABI): per-(request, KV head) dequantization scales,
bfloat16 and float16 queries, the optional terms, unread slots poisoned with
the NaN code, and sampled requests of the full-size batch."""
import pytest
import torch

import oracle
from gqa_softmax_attention_gb300 import workloads as W

from parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gqa_softmax_attention_gb300 import build
    build.build()
    import gqa_softmax_attention_gb300 as m
    yield m
    m.gqa_device_error()


def run(g, p, q=None, scales=True, **kw):
    dev = "cuda"
    q = p["q"] if q is None else q
    ks = p["k_scale"].to(dev) if scales else None
    vs = p["v_scale"].to(dev) if scales else None
    o, lse = g.attn_decode_paged_fp8kv(q.to(dev), p["k_cache"].to(dev), p["v_cache"].to(dev), ks, vs,
                                       p["real_seqlen_kv"].to(dev), p["block_table"].to(dev), **kw)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def reference(p, q=None, scales=True, **kw):
    q = p["q"] if q is None else q
    return oracle.attn_paged_fp8kv(q, p["k_cache"], p["v_cache"], p["k_scale"] if scales else None,
                                   p["v_scale"] if scales else None, p["real_seqlen_kv"], p["block_table"], **kw)


def poison_unread(p):
    """Every cache slot the requests do not own (unused pages, the tail of each
    request's last page) gets the NaN code: results must not change."""
    kc, vc = p["k_cache"].view(torch.uint8).clone(), p["v_cache"].view(torch.uint8).clone()
    ps = kc.shape[1]
    owned = torch.zeros(kc.shape[0], ps, dtype=torch.bool)
    for b, L in enumerate(p["real_seqlen_kv"].tolist()):
        for t in range(L):
            owned[p["block_table"][b, t // ps], t % ps] = True
    kc[~owned] = 0x7F
    vc[~owned] = 0x7F
    return dict(p, k_cache=kc.view(torch.float8_e4m3fn), v_cache=vc.view(torch.float8_e4m3fn))


SMALL = [
    # B, Sq, Hq, Hkv, D, page_size, lengths
    (5, 1, 8, 2, 128, 16, [1, 0, 300, 17, 64]),      # empty request, ragged last pages (16 rows per KV head)
    (4, 4, 24, 2, 256, 16, [3, 700, 129, 2000]),     # 48 rows per KV head; L < Sq
    (2, 1, 64, 1, 128, 64, [1000, 3333]),            # 64 rows per KV head, pages of a whole tile
    (2, 5, 16, 1, 128, 8, [90, 260]),                # 80 rows: two row blocks, 8-token pages
    (1, 1, 2, 1, 256, 32, [5000]),                   # one long request, many splits
    (3, 3, 6, 2, 128, 16, [2, 3, 4]),                # 9 rows, L around Sq
    (2, 2, 32, 4, 128, 128, [50, 401]),              # pages longer than the key tile
    (3, 1, 32, 8, 128, 64, [64, 65, 1]),             # one-key and exact-tile tails
    (2, 3, 64, 1, 128, 64, [700, 1500]),             # 192 rows: the split kernel, three row blocks
    (2, 2, 48, 1, 256, 96, [500, 1000]),             # 96 rows, pages of no 64-key tiling: split, two row blocks
    # page sizes the byte boxes cannot tile: rows gathered with cp.async
    (3, 1, 8, 2, 128, 1, [1, 77, 300]),              # one-token pages
    (2, 4, 24, 2, 256, 5, [3, 901]),                 # 48 rows per KV head (split kernel, not tensor cores)
    (4, 1, 32, 8, 128, 12, [12, 13, 0, 600]),        # 12-token pages, an empty request
    (2, 2, 16, 2, 128, 24, [500, 49]),               # a multiple of 8 that does not tile the 64-key tile
    (2, 2, 16, 4, 128, 64, [100, 2000]),             # 8 rows per KV head (4 heads x 2 queries): the swapped form
    (2, 2, 6, 2, 256, 16, [40, 700]),                # 6 rows per KV head (3 heads x 2 queries), D 256
]


@pytest.mark.parametrize("case", SMALL, ids=[str(c[:6]) for c in SMALL])
def test_small_shapes(g, case):
    B, Sq, Hq, Hkv, D, ps, lengths = case
    p = poison_unread(W.paged_fp8_inputs(B, Sq, Hq, Hkv, D, ps, lengths=lengths, seed=sum(lengths) % 89))
    o, lse = run(g, p)
    ro, rl = reference(p)
    compare(o, lse, ro, rl, str(case))


@pytest.mark.parametrize("Sq", [2, 1], ids=["16rows", "8rows_swapped"])
def test_unit_scales_and_fp16_query(g, Sq):
    p = W.paged_fp8_inputs(3, Sq, 16, 2, 128, 16, lengths=[77, 1, 500], seed=5)
    o, lse = run(g, p, scales=False)
    ro, rl = reference(p, scales=False)
    compare(o, lse, ro, rl, "no scales")
    q16 = p["q"].to(torch.float16)
    o, lse = run(g, p, q=q16)
    assert o.dtype == torch.float16
    ro, rl = reference(p, q=q16)
    compare(o, lse, ro, rl, "float16 query")


def test_scales_reach_the_right_heads(g):
    """Scales spread over two orders of magnitude, different per request and
    KV head: a scale read for the wrong (request, head) would show."""
    p = W.paged_fp8_inputs(4, 2, 16, 4, 128, 16, lengths=[300, 41, 999, 5], seed=6, scale_range=(0.05, 2.0))
    o, lse = run(g, p)
    ro, rl = reference(p)
    compare(o, lse, ro, rl, "spread scales")


@pytest.mark.parametrize("Sq", [4, 2], ids=["16rows", "8rows_swapped"])
@pytest.mark.parametrize("D", [128, 256])
def test_options_and_non_causal(g, D, Sq):
    p = W.paged_fp8_inputs(3, Sq, 8, 2, D, 16, lengths=[300, 17, 1200], seed=7)
    sinks = torch.tensor([0.5, -1.0, float("-inf"), 2.0, 0.0, 1.0, 3.0, -0.5])
    kw = dict(window_left=100, window_right=0, softcap=5.0, sinks=sinks)
    o, lse = run(g, p, **kw)
    ro, rl = reference(p, **kw)
    compare(o, lse, ro, rl, "window + softcap + sinks")
    o, lse = run(g, p, causal=False, scale=0.05)
    ro, rl = reference(p, causal=False, scale=0.05)
    compare(o, lse, ro, rl, "non-causal")


@pytest.mark.parametrize("D", [128, 256])
def test_wide_groups_options_and_fp16(g, D):
    """32-128 rows per KV head take the tensor-core decode with widened tiles:
    window + softcap + sinks, non-causal, and a float16 query there."""
    p = W.paged_fp8_inputs(3, 4, 24, 2, D, 16, lengths=[700, 5, 2100], seed=11, scale_range=(0.1, 1.5))
    sinks = torch.linspace(-2.0, 2.0, 24)
    sinks[3] = float("-inf")
    kw = dict(window_left=300, window_right=0, softcap=6.0, sinks=sinks)
    o, lse = run(g, p, **kw)
    ro, rl = reference(p, **kw)
    compare(o, lse, ro, rl, "tc: window + softcap + sinks")
    o, lse = run(g, p, causal=False, scale=0.04)
    ro, rl = reference(p, causal=False, scale=0.04)
    compare(o, lse, ro, rl, "tc: non-causal")
    q16 = p["q"].to(torch.float16)
    o, lse = run(g, p, q=q16)
    ro, rl = reference(p, q=q16)
    compare(o, lse, ro, rl, "tc: float16 query")


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("Hq", [16, 40, 64], ids=["32rows", "80rows", "128rows"])
def test_tensor_core_widener_teams(g, D, Hq):
    """The tensor-core decode's widening warps split into a K and a V team whose
    sizes follow the rows per KV head (32: three K warps and two V, 80: one and
    two, 128: one and one); ragged tails and unread slots poisoned with NaN."""
    p = poison_unread(W.paged_fp8_inputs(3, 4, Hq, 2, D, 16, lengths=[5, 333, 1500], seed=17))
    o, lse = run(g, p)
    ro, rl = reference(p)
    compare(o, lse, ro, rl, "tc teams")


def test_matches_16bit_path_on_widened_cache(g):
    """The FP8 call equals the 16-bit decode on the caches widened to float16
    (every e4m3fn value is a float16), unit scales, float16 query."""
    p = W.paged_fp8_inputs(3, 1, 32, 8, 128, 64, lengths=[2000, 64, 513], seed=8)
    q16 = p["q"].to(torch.float16)
    o8, l8 = run(g, p, q=q16, scales=False)
    dev = "cuda"
    o16, l16 = g.decode_paged(q16.to(dev), p["k_cache"].to(torch.float16).to(dev),
                              p["v_cache"].to(torch.float16).to(dev), p["real_seqlen_kv"].to(dev),
                              p["block_table"].to(dev))
    compare(o8, l8, o16.cpu().double(), l16.cpu().double(), "fp8 vs fp16 path")


@pytest.mark.parametrize("name", ["paged_decode_fp8kv", "wide_group_decode_fp8kv"])
def test_full_size_workload(g, name):
    p = W.make(name)
    o, lse = run(g, p)
    L = p["real_seqlen_kv"]
    order = torch.argsort(L)
    gen = torch.Generator().manual_seed(0)
    mid = order[1:-1][torch.randperm(len(order) - 2, generator=gen)[:6]]
    reqs = sorted({int(order[0]), int(order[-1])} | set(mid.tolist()))
    ro, rl = oracle.attn_paged_fp8kv(p["q"], p["k_cache"], p["v_cache"], p["k_scale"], p["v_scale"], L,
                                     p["block_table"], requests=reqs)
    sel = torch.tensor(reqs)
    compare(o[sel], lse[sel], ro[sel], rl[sel], name)
    assert not torch.isnan(o.float()).any() and bool(torch.isfinite(lse).all())
