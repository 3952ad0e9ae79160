"""Sliding window, softcap and sinks on the GPU against the FP64 oracle.

The optional terms of TileOPs "Attention Operators" (GQADenseFwdOp stages 5-6,
GQAPagedFwdOp's sinks), through the C ABI's _ex entry points, for the dense
prefill kernel and every paged decode path (split kernels with TMA page boxes
or cp.async gathers, the balanced tensor-core kernel).
"""
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
    m.gqa_device_error()


def sinks_for(Hq, seed, with_inf=False):
    gen = torch.Generator().manual_seed(seed)
    s = torch.randn(Hq, generator=gen) * 2.0
    s[0] = -INF                                   # a disabled sink
    if with_inf:
        s[-1] = INF                               # a head whose output is zero
    return s


def check(o, lse, ro, rl, label):
    """compare(), with rows whose reference LSE is +inf (a +inf sink) checked
    apart: zero output and LSE +inf."""
    pos = torch.isposinf(rl)
    if bool(pos.any()):
        assert bool(torch.all(torch.isposinf(lse.cpu()[pos]))), label + ": LSE of a +inf sink row"
        assert bool(torch.all(o.float().cpu()[pos] == 0)), label + ": output of a +inf sink row"
        keep = ~pos
        o, lse, ro, rl = o.cpu()[keep], lse.cpu()[keep], ro[keep], rl[keep]
    return compare(o, lse, ro, rl, label)


DENSE = [
    # B, Hq, Hkv, Sq, Skv, D, causal, window_left, window_right, softcap, sinks, mask
    (1, 4, 2, 200, 200, 128, True, 0, -1, 0.0, False, None),        # one key per row
    (2, 8, 2, 300, 700, 128, True, 128, -1, 0.0, False, None),      # window across tiles, chunked shape
    (1, 4, 2, 257, 513, 64, True, 300, -1, 20.0, True, None),
    (2, 4, 1, 190, 400, 128, False, 50, 70, 0.0, False, 0.7),       # two-sided window, padding
    (1, 8, 2, 256, 256, 128, True, -1, -1, 5.0, False, None),       # softcap alone
    (2, 4, 2, 129, 260, 64, True, -1, -1, 0.0, True, 0.8),          # sinks alone (+inf head)
    (1, 16, 2, 512, 1024, 128, True, 700, -1, 30.0, True, None),
]


@pytest.mark.parametrize("case", DENSE, ids=[str(c) for c in DENSE])
def test_dense_options(g, case):
    B, Hq, Hkv, Sq, Skv, D, causal, wl, wr, cap, sk, mk = case
    d = W.dense_inputs(B, Hq, Hkv, Sq, Skv, D, seed=Sq + 3 * Skv)
    mask = None
    if mk is not None:
        gen = torch.Generator().manual_seed(5)
        mask = torch.rand(B, Skv, generator=gen) < mk
    sinks = sinks_for(Hq, Sq, with_inf=sk) if sk else None
    o, lse = g.attention(d["q"].cuda(), d["k"].cuda(), d["v"].cuda(), causal=causal,
                         key_padding_mask=mask.cuda() if mask is not None else None, window_left=wl,
                         window_right=wr, softcap=cap, sinks=sinks.cuda() if sinks is not None else None)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_dense(d["q"], d["k"], d["v"], key_padding_mask=mask, causal=causal, window_left=wl,
                               window_right=wr, softcap=cap, sinks=sinks)
    check(o, lse, ro, rl, str(case))


PAGED = [
    # B, Sq, Hq, Hkv, D, page_size, lengths, window_left, softcap, sinks       (rows per KV head -> path)
    (5, 1, 8, 2, 128, 16, [1, 0, 300, 17, 2000], 100, 0.0, False),    # 4 rows: split kernel, TMA pages
    (3, 2, 32, 4, 128, 3, [50, 401, 1000], 64, 10.0, True),          # 16 rows: split kernel, gathered pages
    (4, 4, 24, 2, 256, 16, [3, 700, 129, 3000], 257, 0.0, True),      # 48 rows: tensor-core kernel
    (2, 4, 32, 1, 128, 64, [129, 5000], 1000, 25.0, False),           # 128 rows: tensor-core kernel
    (3, 1, 8, 2, 128, 64, [5000, 64, 900], -1, 15.0, True),           # softcap + sinks, no window
    (2, 2, 16, 1, 64, 8, [7000, 300], 10, 0.0, False),                # narrow window, many splits
]


@pytest.mark.parametrize("case", PAGED, ids=[str(c[:6]) for c in PAGED])
def test_paged_options(g, case):
    B, Sq, Hq, Hkv, D, ps, lengths, wl, cap, sk = case
    p = W.paged_inputs(B, Sq, Hq, Hkv, D, ps, lengths=lengths, seed=sum(lengths) % 89)
    sinks = sinks_for(Hq, B + Sq, with_inf=True) if sk else None
    o, lse = g.decode_paged(p["q"].cuda(), p["k_cache"].cuda(), p["v_cache"].cuda(), p["real_seqlen_kv"].cuda(),
                            p["block_table"].cuda(), window_left=wl, softcap=cap,
                            sinks=sinks.cuda() if sinks is not None else None)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_paged(p["q"], p["k_cache"], p["v_cache"], p["real_seqlen_kv"], p["block_table"],
                               window_left=wl, softcap=cap, sinks=sinks)
    check(o, lse, ro, rl, str(case))


def test_window_reads_less_cache(g):
    """A left window bounds what decode reads: poisoning every cache slot left
    of all windows with NaN leaves the result unchanged (and equal to the
    oracle on clean data)."""
    B, Sq, Hq, Hkv, D, ps, wl = 2, 4, 24, 2, 256, 16, 200
    p = W.paged_inputs(B, Sq, Hq, Hkv, D, ps, lengths=[3000, 1500], seed=9)
    ro, rl = oracle.attn_paged(p["q"], p["k_cache"], p["v_cache"], p["real_seqlen_kv"], p["block_table"],
                               window_left=wl)
    kc, vc = p["k_cache"].clone(), p["v_cache"].clone()
    for b, L in enumerate(p["real_seqlen_kv"].tolist()):
        first_visible = L - Sq - wl
        for t in range(max(0, first_visible // 64 * 64)):
            kc[p["block_table"][b, t // ps], t % ps] = float("nan")
            vc[p["block_table"][b, t // ps], t % ps] = float("nan")
    o, lse = g.decode_paged(p["q"].cuda(), kc.cuda(), vc.cuda(), p["real_seqlen_kv"].cuda(),
                            p["block_table"].cuda(), window_left=wl)
    torch.cuda.synchronize()
    check(o, lse, ro, rl, "poisoned left of the window")
