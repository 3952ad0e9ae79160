"""The paged calls keep their metadata on the device and allocate nothing when
given their buffers, so they can be captured in a CUDA graph once and
replayed with new lengths and tables (TileOPs GQAPagedFwdOp: device lengths
stay live replay inputs; choosing and preparing the path needs no host
read-back).  Each replay is checked against the FP64 oracle."""
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


def test_paged_decode_graph_replay(g):
    B, Sq, Hq, Hkv, D, ps = 8, 1, 32, 8, 128, 64
    p = W.paged_inputs(B, Sq, Hq, Hkv, D, ps, lengths=[4000] * B, seed=1)
    dev = {n: p[n].cuda() for n in ("q", "k_cache", "v_cache", "real_seqlen_kv", "block_table")}
    ws = torch.empty(g.attn_decode_paged_workspace_size(B, Sq, Hq, Hkv, D, ps, p["block_table"].shape[1]),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty_like(dev["q"])
    lse = torch.empty((B, Sq, Hq), dtype=torch.float32, device="cuda")
    run = lambda: g.decode_paged(dev["q"], dev["k_cache"], dev["v_cache"], dev["real_seqlen_kv"],
                                 dev["block_table"], causal=True, workspace=ws, out=out, lse=lse)
    run()                                      # first call outside capture (loads the library, sets attributes)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    gen = torch.Generator().manual_seed(2)
    for _ in range(3):
        lens = torch.randint(1, 4001, (B,), generator=gen, dtype=torch.int32)
        dev["real_seqlen_kv"].copy_(lens)
        graph.replay()
        torch.cuda.synchronize()
        ro, rl = oracle.attn_paged(p["q"], p["k_cache"], p["v_cache"], lens, p["block_table"], causal=True)
        compare(out.cpu(), lse.cpu(), ro, rl, "decode replay")


@pytest.mark.parametrize("split_decode", [False, True], ids=["packed_only", "split_decode"])
def test_mixed_paged_graph_replay(g, split_decode):
    """A mixed call replays with new cache lengths and a new query split; with
    the larger workspace its one-query requests (which change between
    replays) run on the split decode kernel."""
    ql, L = [1, 300, 1, 4], [2000, 700, 50, 1000]
    Hq, Hkv, D, ps = 8, 2, 128, 16
    p = W.varlen_paged_inputs(ql, L, Hq, Hkv, D, ps, seed=4)
    names = ("q", "k_cache", "v_cache", "cu_seqlens_q", "cache_seqlens", "block_table")
    dev = {n: p[n].cuda() for n in names}
    tq = p["q"].shape[0]
    size = (g.attn_paged_workspace_size(len(ql), tq, Hq, Hkv, D, ps, p["block_table"].shape[1]) if split_decode
            else g.attn_varlen_workspace_size(len(ql), tq, Hq, Hkv))
    ws = torch.empty(size, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(dev["q"])
    lse = torch.empty((p["q"].shape[0], Hq), dtype=torch.float32, device="cuda")
    run = lambda: g.paged(*[dev[n] for n in names], causal=True, out=out, lse=lse, workspace=ws)
    run()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    # new cache lengths (still >= each request's query count) and a new query split
    for lens, cu in (([2000, 700, 50, 1000], [0, 1, 301, 302, 306]), ([17, 400, 1, 999], [0, 1, 301, 302, 306]),
                     ([1500, 305, 30, 10], [0, 0, 300, 302, 306])):
        dev["cache_seqlens"].copy_(torch.tensor(lens, dtype=torch.int32))
        dev["cu_seqlens_q"].copy_(torch.tensor(cu, dtype=torch.int32))
        graph.replay()
        torch.cuda.synchronize()
        ro, rl = oracle.attn_paged_varlen(p["q"], p["k_cache"], p["v_cache"], torch.tensor(cu, dtype=torch.int32),
                                          torch.tensor(lens, dtype=torch.int32), p["block_table"], causal=True)
        compare(out.cpu(), lse.cpu(), ro, rl, "mixed replay %s" % lens)


def _mixed_case(seed):
    ql, L = [1, 600, 1, 1, 300], [3000, 1800, 40, 7000, 700]
    Hq, Hkv, D, ps = 32, 8, 128, 64
    p = W.varlen_paged_inputs(ql, L, Hq, Hkv, D, ps, seed=seed)
    names = ("q", "k_cache", "v_cache", "cu_seqlens_q", "cache_seqlens", "block_table")
    dev = {n: p[n].cuda() for n in names}
    return p, names, dev, (len(ql), p["q"].shape[0], Hq, Hkv, D, ps, p["block_table"].shape[1])


def test_mixed_paged_on_side_stream_then_caller_work(g):
    """A mixed call on a non-default stream runs its chunks on the library's
    side stream and joins back: work queued on the caller's stream right after
    the call (here a copy of the outputs) sees both parts complete."""
    p, names, dev, sz = _mixed_case(6)
    ws = torch.empty(g.attn_paged_workspace_size(*sz), dtype=torch.uint8, device="cuda")
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for _ in range(3):
            out, lse = g.paged(*[dev[n] for n in names], causal=True, workspace=ws)
            o_copy, l_copy = out.clone(), lse.clone()     # queued on st behind the call
    torch.cuda.synchronize()
    ro, rl = oracle.attn_paged_varlen(p["q"], p["k_cache"], p["v_cache"], p["cu_seqlens_q"], p["cache_seqlens"],
                                      p["block_table"], causal=True)
    compare(o_copy.cpu(), l_copy.cpu(), ro, rl, "mixed call on a side stream, copied on the caller's stream")


def test_mixed_paged_captured_in_fresh_thread(g):
    """Captured in a host thread that has made no earlier mixed call (no side
    stream yet, and none may be created during a capture): the call runs both
    parts on the capturing stream, and the graph replays correctly."""
    import threading
    p, names, dev, sz = _mixed_case(8)
    ws = torch.empty(g.attn_paged_workspace_size(*sz), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(dev["q"])
    lse = torch.empty((p["q"].shape[0], 32), dtype=torch.float32, device="cuda")
    err = []

    def body():
        try:
            torch.cuda.set_device(0)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                g.paged(*[dev[n] for n in names], causal=True, out=out, lse=lse, workspace=ws)
            graph.replay()
            torch.cuda.synchronize()
        except Exception as e:          # reported in the main thread
            err.append(e)

    t = threading.Thread(target=body)
    t.start()
    t.join()
    assert not err, err
    ro, rl = oracle.attn_paged_varlen(p["q"], p["k_cache"], p["v_cache"], p["cu_seqlens_q"], p["cache_seqlens"],
                                      p["block_table"], causal=True)
    compare(out.cpu(), lse.cpu(), ro, rl, "mixed call captured in a fresh thread")


def test_fp8kv_decode_graph_replay(g):
    """The FP8-KV decode replays with new lengths and new scales."""
    B, Sq, Hq, Hkv, D, ps = 6, 1, 32, 8, 128, 64
    p = W.paged_fp8_inputs(B, Sq, Hq, Hkv, D, ps, lengths=[3000] * B, seed=9)
    dev = {n: p[n].cuda() for n in ("q", "k_cache", "v_cache", "k_scale", "v_scale", "real_seqlen_kv",
                                    "block_table")}
    ws = torch.empty(g.attn_decode_paged_workspace_size(B, Sq, Hq, Hkv, D, ps, p["block_table"].shape[1]),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty_like(dev["q"])
    lse = torch.empty((B, Sq, Hq), dtype=torch.float32, device="cuda")
    run = lambda: g.attn_decode_paged_fp8kv(dev["q"], dev["k_cache"], dev["v_cache"], dev["k_scale"], dev["v_scale"],
                                            dev["real_seqlen_kv"], dev["block_table"], causal=True, workspace=ws,
                                            out=out, lse=lse)
    run()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    gen = torch.Generator().manual_seed(10)
    for _ in range(3):
        lens = torch.randint(1, 3001, (B,), generator=gen, dtype=torch.int32)
        ks = torch.rand(B, Hkv, generator=gen) + 0.1
        vs = torch.rand(B, Hkv, generator=gen) + 0.1
        dev["real_seqlen_kv"].copy_(lens)
        dev["k_scale"].copy_(ks)
        dev["v_scale"].copy_(vs)
        graph.replay()
        torch.cuda.synchronize()
        ro, rl = oracle.attn_paged_fp8kv(p["q"], p["k_cache"], p["v_cache"], ks, vs, lens, p["block_table"],
                                         causal=True)
        compare(out.cpu(), lse.cpu(), ro, rl, "fp8 decode replay")
