"""Paged decode on the GPU against the FP64 oracle (through the C ABI)."""
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


def run(g, p, causal=True, scale=None):
    dev = "cuda"
    o, lse = g.decode_paged(p["q"].to(dev), p["k_cache"].to(dev), p["v_cache"].to(dev),
                            p["real_seqlen_kv"].to(dev), p["block_table"].to(dev), causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def poison_unread(p):
    """Fill every cache slot the requests do not own (unused pages and the
    tail of each request's last page) with NaN: results must not change."""
    kc, vc = p["k_cache"].clone(), p["v_cache"].clone()
    ps = kc.shape[1]
    owned = torch.zeros(kc.shape[0], ps, dtype=torch.bool)
    for b, L in enumerate(p["real_seqlen_kv"].tolist()):
        for t in range(L):
            owned[p["block_table"][b, t // ps], t % ps] = True
    kc[~owned] = float("nan")
    vc[~owned] = float("nan")
    return dict(p, k_cache=kc, v_cache=vc)


SMALL = [
    # B, Sq, Hq, Hkv, D, page_size, lengths
    (5, 1, 8, 2, 128, 16, [1, 0, 300, 17, 64]),      # empty request, ragged last pages
    (3, 1, 4, 4, 64, 1, [5, 40, 2]),                 # page size 1, MHA (one row per CTA)
    (4, 4, 24, 2, 256, 16, [3, 700, 129, 2000]),     # 48 rows per KV head; L < Sq
    (2, 2, 32, 4, 128, 3, [50, 401]),                # page size 3 (not a power of two), 16 rows
    (2, 1, 64, 1, 128, 64, [1000, 3333]),            # 64 rows per KV head
    (2, 5, 16, 1, 64, 8, [90, 260]),                 # 80 rows: two row blocks
    (1, 1, 2, 1, 256, 32, [5000]),                   # one long request, many splits
    (3, 3, 6, 2, 128, 16, [2, 3, 4]),                # 9 rows, L around Sq
    # 32..128 packed rows per KV head: the tensor-core decode kernel
    (3, 4, 16, 2, 128, 32, [4100, 3, 700]),          # 32 rows, L < Sq, ragged tail
    (2, 4, 32, 1, 128, 16, [129, 2000]),             # 128 rows
    (4, 2, 48, 1, 256, 64, [64, 65, 0, 999]),        # 96 rows, empty request, one-key tile
    (2, 4, 24, 2, 256, 8, [1, 5000]),                # 48 rows, 8-token pages
    (3, 4, 16, 2, 256, 16, [5, 333, 1500]),          # 32 rows at D 256 (one softmax warp)
    (2, 4, 64, 2, 256, 32, [700, 1201]),             # 128 rows at D 256 (four softmax warps)
]


@pytest.mark.parametrize("case", SMALL, ids=[str(c[:6]) for c in SMALL])
def test_small_shapes(g, case):
    B, Sq, Hq, Hkv, D, ps, lengths = case
    p = W.paged_inputs(B, Sq, Hq, Hkv, D, ps, lengths=lengths, seed=sum(lengths) % 97)
    p = poison_unread(p)
    o, lse = run(g, p)
    ro, rl = oracle.attn_paged(p["q"], p["k_cache"], p["v_cache"], p["real_seqlen_kv"], p["block_table"])
    compare(o, lse, ro, rl, str(case))


@pytest.mark.parametrize("shape", [(3, 4, 8, 2, 128, 16), (2, 4, 24, 2, 256, 16)], ids=["rows16", "rows48"])
def test_non_causal_and_scale(g, shape):
    B, Sq, Hq, Hkv, D, ps = shape
    p = W.paged_inputs(B, Sq, Hq, Hkv, D, ps, lengths=[10, 0, 77][:B] if B == 3 else [300, 17], seed=3)
    o, lse = run(g, p, causal=False, scale=0.05)
    ro, rl = oracle.attn_paged(p["q"], p["k_cache"], p["v_cache"], p["real_seqlen_kv"], p["block_table"],
                               causal=False, scale=0.05)
    compare(o, lse, ro, rl, "non-causal")


def test_paged_matches_dense_gpu(g):
    """Gather the pool per request and run the dense kernel: the two GPU paths agree."""
    p = W.paged_inputs(3, 2, 16, 4, 128, 16, lengths=[300, 1, 513], seed=8)
    o, lse = run(g, p)
    ps = p["page_size"]
    for b, L in enumerate(p["real_seqlen_kv"].tolist()):
        idx = torch.arange(L)
        phys = p["block_table"][b, idx // ps].long()
        k = p["k_cache"][phys, idx % ps][None].contiguous()
        v = p["v_cache"][phys, idx % ps][None].contiguous()
        od, ld = g.attention(p["q"][b:b + 1].cuda(), k.cuda(), v.cuda(), causal=True)
        compare(o[b:b + 1], lse[b:b + 1], od.cpu().double(), ld.cpu().double(), "request %d" % b)


def test_validate_paged(g):
    p = W.paged_inputs(2, 1, 8, 2, 128, 16, lengths=[40, 3], seed=1)
    sl, bt = p["real_seqlen_kv"].cuda(), p["block_table"].cuda()
    g.attn_validate_paged(sl, bt, 1, 16, p["num_pages"])
    bad = bt.clone()
    bad[0, 1] = p["num_pages"]
    with pytest.raises(ValueError):
        g.attn_validate_paged(sl, bad, 1, 16, p["num_pages"])
    with pytest.raises(ValueError):
        g.attn_validate_paged(torch.tensor([40, 10_000], dtype=torch.int32, device="cuda"), bt, 1, 16,
                              p["num_pages"])


@pytest.mark.parametrize("name,nreq", [("paged_decode", 8), ("wide_group_decode", 6)])
def test_full_size_workload(g, name, nreq):
    p = W.make(name)
    o, lse = run(g, p)
    L = p["real_seqlen_kv"]
    order = torch.argsort(L)
    # the shortest, the longest, and a seeded sample in between
    gen = torch.Generator().manual_seed(0)
    mid = order[1:-1][torch.randperm(len(order) - 2, generator=gen)[:nreq - 2]]
    reqs = sorted({int(order[0]), int(order[-1])} | set(mid.tolist()))
    ro, rl = oracle.attn_paged(p["q"], p["k_cache"], p["v_cache"], L, p["block_table"], requests=reqs)
    sel = torch.tensor(reqs)
    compare(o[sel], lse[sel], ro[sel], rl[sel], name)
    assert not torch.isnan(o.float()).any() and bool(torch.isfinite(lse).all())
