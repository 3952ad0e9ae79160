"""The paged-decode entry point that allocates nothing (attn_decode_paged_noalloc).

It serves callers that cannot allocate device memory or pass a workspace (a
serving engine whose memory is all pre-reserved by its own pool, a plugin in a
host framework that forbids allocation while it runs, a loop that cannot pay
for cudaMalloc's implicit synchronisation): its split partials live in a fixed
array inside the library.  Here it is called through the C ABI and must match
attn_decode_paged (caller workspace) within the parity tolerances, with each
of its two decode routes called twice in a row on different inputs, so a stale
array from the first call would show.  This file sorts last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

from gqa_softmax_attention_gb300 import workloads as W

from parity import TOL_LSE, TOL_MAX, TOL_MEAN

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gqa_softmax_attention_gb300 import _lib, build
    build.build()
    return _lib.load()


def _call(lib, fn, p, extra=()):
    dev = "cuda"
    q = p["q"].to(dev)
    kc, vc = p["k_cache"].to(dev), p["v_cache"].to(dev)
    sl, bt = p["real_seqlen_kv"].to(dev), p["block_table"].to(dev)
    B, Sq, Hq, D = q.shape
    num_pages, ps, Hkv, _ = kc.shape
    o = torch.full((B, Sq, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((B, Sq, Hq), float("nan"), dtype=torch.float32, device=dev)
    st = fn(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kc.data_ptr()), ctypes.c_void_p(vc.data_ptr()),
            ctypes.c_void_p(sl.data_ptr()), ctypes.c_void_p(bt.data_ptr()), ps, ctypes.c_void_p(o.data_ptr()),
            ctypes.c_void_p(lse.data_ptr()), B, Sq, Hq, Hkv, D, num_pages, bt.shape[1], 1, D ** -0.5, *extra,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st, o.cpu(), lse.cpu()


def _with_workspace(lib, p):
    c = p["q"].shape
    need = lib.attn_decode_paged_workspace_size(c[0], c[1], c[2], p["k_cache"].shape[2], c[3], p["page_size"],
                                                p["max_pages"])
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    return _call(lib, lib.attn_decode_paged, p, (ctypes.c_void_p(ws.data_ptr()), ctypes.c_size_t(need)))


def _close(a, b):
    oa, la = a[1].float().double(), a[2].double()
    ob, lb = b[1].float().double(), b[2].double()
    assert torch.equal(torch.isneginf(la), torch.isneginf(lb))
    fin = ~torch.isneginf(lb)
    d = (oa - ob)[fin].abs()
    assert float(d.max()) <= TOL_MAX and float(d.mean()) <= TOL_MEAN
    assert float((la - lb)[fin].abs().max()) <= TOL_LSE
    assert bool(torch.all(oa[~fin] == 0))


def test_noalloc_matches_workspace_entry_point_twice(lib):
    # Each of the two decode routes runs twice in a row on the shared array,
    # the second call with other inputs and shorter requests (one of them
    # empty), so partials or segment-table entries left by the first call
    # would show in the second.
    split_path = [  # 4 query rows per KV head: the split-KV kernel and its partials
        W.paged_inputs(6, 1, 32, 8, 128, 64, lengths=[1500, 0, 7000, 64, 3333, 12000], seed=11),
        W.paged_inputs(5, 1, 32, 8, 128, 64, lengths=[700, 9000, 0, 1, 2100], seed=13),
    ]
    tensor_core_path = [  # 48 rows per KV head: the balanced tensor-core kernel and its segment table
        W.paged_inputs(3, 4, 24, 2, 256, 16, lengths=[900, 2, 5000], seed=12),
        W.paged_inputs(4, 4, 24, 2, 256, 16, lengths=[300, 0, 4, 1200], seed=14),
    ]
    for p in split_path + tensor_core_path:
        na = _call(lib, lib.attn_decode_paged_noalloc, p)
        assert na[0] == 0, lib.gqa_status_string(na[0])
        ref = _with_workspace(lib, p)
        assert ref[0] == 0
        _close(na, ref)


def test_noalloc_python_wrapper_checks_its_arguments(lib):
    import gqa_softmax_attention_gb300 as g
    p = W.paged_inputs(2, 1, 8, 2, 128, 16, lengths=[40, 17], seed=15)
    dev = "cuda"
    q, kc, vc = p["q"].to(dev), p["k_cache"].to(dev), p["v_cache"].to(dev)
    sl, bt = p["real_seqlen_kv"].to(dev), p["block_table"].to(dev)
    o, lse = g.attn_decode_paged_noalloc(q, kc, vc, sl, bt)
    ref = _with_workspace(lib, p)
    torch.cuda.synchronize()
    _close((0, o.cpu(), lse.cpu()), ref)
    bad = [
        dict(real_seqlen_kv=sl.cpu()),                       # lengths on the host
        dict(block_table=bt.to(torch.int64)),                # wrong index type
        dict(v_cache=vc[:, :8].contiguous()),                # smaller value cache
        dict(k_cache=kc[..., :64].contiguous()),             # head dim differs from q's
        dict(real_seqlen_kv=sl[:1]),                         # not [B]
    ]
    for change in bad:
        args = dict(q=q, k_cache=kc, v_cache=vc, real_seqlen_kv=sl, block_table=bt)
        args.update(change)
        with pytest.raises(ValueError):
            g.attn_decode_paged_noalloc(**args)
    # a strided block table is made contiguous, not read with the wrong stride
    wide = torch.full((bt.shape[0], 2 * bt.shape[1]), -1, dtype=torch.int32, device=dev)
    wide[:, ::2] = bt
    o2, lse2 = g.attn_decode_paged_noalloc(q, kc, vc, sl, wide[:, ::2])
    torch.cuda.synchronize()
    _close((0, o2.cpu(), lse2.cpu()), ref)


def test_noalloc_refuses_sizes_beyond_its_array(lib):
    cap = lib.attn_decode_paged_noalloc_max_workspace()
    assert cap == 32 << 20
    # 24/2/D256 decode over 32K-token requests needs far more than 32 MiB of partials
    B, Sq, Hq, Hkv, D, ps, max_pages = 64, 4, 24, 2, 256, 16, 2048
    assert lib.attn_decode_paged_workspace_size(B, Sq, Hq, Hkv, D, ps, max_pages) > cap
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    ptr = ctypes.c_void_p(z.data_ptr())
    st = lib.attn_decode_paged_noalloc(ptr, ptr, ptr, ptr, ptr, ps, ptr, None, B, Sq, Hq, Hkv, D, 1, max_pages, 1,
                                       0.1, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 4      # GQA_ERR_WORKSPACE, nothing launched
