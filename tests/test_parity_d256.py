"""Dense prefill with head dim 256 (one query tile per CTA) against the FP64
oracle, through the C ABI: the 24/2/D256 geometry of MATE "QSA" as a dense
causal prefill, ragged tails, chunked and Sq > Skv shapes, padding masks,
the optional terms of TileOPs GQADenseFwdOp and float16 inputs."""
import pytest
import torch

import oracle
from gqa_softmax_attention_gb300 import workloads as W

from parity import compare, sample_rows

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


def masks(kind, B, Skv, seed):
    if kind is None:
        return None
    if kind == "prefix":                      # batch 1 has no key at all
        return torch.arange(Skv)[None, :] < torch.tensor([[Skv // 3], [0]])[:B]
    if kind == "runs":                        # long fully padded stretches: skipped tiles
        m = torch.zeros(B, Skv, dtype=torch.bool)
        m[:, 5:9] = True
        m[:, 600:900] = True
        return m
    gen = torch.Generator().manual_seed(seed)
    return torch.rand(B, Skv, generator=gen) < kind


SMALL = [
    # B, Hq, Hkv, Sq, Skv, causal, mask, scale
    (1, 4, 2, 128, 128, True, None, None),
    (1, 24, 2, 200, 200, True, None, None),          # ragged tail, g = 12
    (2, 4, 1, 300, 700, True, None, None),           # chunked prefill shape
    (2, 6, 3, 257, 129, True, None, None),           # Sq > Skv: leading rows empty
    (2, 4, 2, 130, 390, False, 0.5, None),           # random padding, non-causal
    (2, 8, 2, 256, 384, True, "prefix", None),       # prefix padding, one batch empty
    (1, 2, 1, 64, 1000, False, "runs", None),        # tile skipping
    (1, 4, 2, 190, 190, True, None, 0.0),            # scale 0: mean of visible values
    (1, 4, 4, 5, 3, True, None, None),               # fewer keys than a tile, MHA
]


@pytest.mark.parametrize("case", SMALL, ids=[str(c) for c in SMALL])
def test_small_shapes(g, case):
    B, Hq, Hkv, Sq, Skv, causal, mk, scale = case
    d = W.dense_inputs(B, Hq, Hkv, Sq, Skv, 256, seed=Sq + 7 * Skv)
    mask = masks(mk, B, Skv, seed=Sq)
    o, lse = g.attention(d["q"].cuda(), d["k"].cuda(), d["v"].cuda(), causal=causal, scale=scale,
                         key_padding_mask=mask.cuda() if mask is not None else None)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_dense(d["q"], d["k"], d["v"], key_padding_mask=mask, causal=causal, scale=scale)
    compare(o, lse, ro, rl, str(case))


def test_many_items_per_cta(g):
    """More work items than CTAs (the persistent loop wraps several times,
    items of different lengths alternate): sampled rows against the oracle."""
    B, Hq, Hkv, S = 2, 24, 2, 1536                  # 12 query tiles x 48 heads = 576 items
    d = W.dense_inputs(B, Hq, Hkv, S, S, 256, seed=11)
    o, lse = g.attention(d["q"].cuda(), d["k"].cuda(), d["v"].cuda(), causal=True)
    torch.cuda.synchronize()
    rows = sample_rows(B, S, Hq, extra=160, seed=3)
    ro, rl = oracle.attn_dense_rows(d["q"], d["k"], d["v"], rows, causal=True)
    idx = torch.tensor(rows)
    compare(o.cpu()[idx[:, 0], idx[:, 1], idx[:, 2]], lse.cpu()[idx[:, 0], idx[:, 1], idx[:, 2]], ro, rl,
            "many items")


def test_single_visible_key_is_exact(g):
    d = W.dense_inputs(1, 4, 2, 140, 140, 256, seed=5)
    o, lse = g.attention(d["q"].cuda(), d["k"].cuda(), d["v"].cuda(), causal=True, scale=0.25)
    o = o.cpu()
    for h in range(4):
        assert torch.equal(o[0, 0, h], d["v"][0, 0, h // 2])


def test_gqa_equals_repeated_kv(g):
    d = W.dense_inputs(1, 8, 2, 256, 256, 256, seed=4)
    o, lse = g.attention(d["q"].cuda(), d["k"].cuda(), d["v"].cuda(), causal=True)
    rep_k = d["k"].repeat_interleave(4, dim=2).contiguous().cuda()
    rep_v = d["v"].repeat_interleave(4, dim=2).contiguous().cuda()
    o2, l2 = g.attention(d["q"].cuda(), rep_k, rep_v, causal=True)
    assert torch.equal(o, o2) and torch.equal(lse, l2)


OPTIONS = [
    # B, Hq, Hkv, Sq, Skv, causal, window_left, window_right, softcap, sinks
    (1, 4, 2, 200, 200, True, 0, -1, 0.0, False),        # one key per row
    (2, 8, 2, 300, 700, True, 128, -1, 0.0, False),      # window across tiles
    (2, 4, 1, 190, 400, False, 50, 70, 20.0, False),     # two-sided window, softcap
    (1, 12, 2, 256, 256, True, -1, -1, 0.0, True),       # sinks (+inf head, -inf head)
]


@pytest.mark.parametrize("case", OPTIONS, ids=[str(c) for c in OPTIONS])
def test_options(g, case):
    B, Hq, Hkv, Sq, Skv, causal, wl, wr, cap, sk = case
    d = W.dense_inputs(B, Hq, Hkv, Sq, Skv, 256, seed=Skv)
    sinks = None
    if sk:
        gen = torch.Generator().manual_seed(Sq)
        sinks = torch.randn(Hq, generator=gen) * 2.0
        sinks[0], sinks[-1] = -INF, INF
    o, lse = g.attention(d["q"].cuda(), d["k"].cuda(), d["v"].cuda(), causal=causal, window_left=wl,
                         window_right=wr, softcap=cap, sinks=sinks.cuda() if sinks is not None else None)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_dense(d["q"], d["k"], d["v"], causal=causal, window_left=wl, window_right=wr,
                               softcap=cap, sinks=sinks)
    o, lse = o.cpu(), lse.cpu()
    pos = torch.isposinf(rl)
    if bool(pos.any()):                       # a +inf sink: zero output, LSE +inf
        assert bool(torch.all(torch.isposinf(lse[pos]))) and bool(torch.all(o.float()[pos] == 0))
        o, lse, ro, rl = o[~pos], lse[~pos], ro[~pos], rl[~pos]
    compare(o, lse, ro, rl, str(case))


def test_float16(g):
    d = W.dense_inputs(2, 8, 2, 300, 300, 256, seed=8)
    q, k, v = (d[n].to(torch.float16) for n in ("q", "k", "v"))
    o, lse = g.attention(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert o.dtype == torch.float16
    ro, rl = oracle.attn_dense(q, k, v, causal=True)
    compare(o, lse, ro, rl, "float16")


def test_full_size_workload_sampled_rows(g):
    d = W.make("wide_group_prefill")
    cfg = d["config"]
    o, lse = g.attention(d["q"].cuda(), d["k"].cuda(), d["v"].cuda(), causal=True)
    torch.cuda.synchronize()
    o, lse = o.cpu(), lse.cpu()
    rows = sample_rows(cfg["B"], cfg["Sq"], cfg["Hq"], extra=64)
    ro, rl = oracle.attn_dense_rows(d["q"], d["k"], d["v"], rows, causal=True)
    idx = torch.tensor(rows)
    compare(o[idx[:, 0], idx[:, 1], idx[:, 2]], lse[idx[:, 0], idx[:, 1], idx[:, 2]], ro, rl, "wide_group_prefill")
    assert not torch.isnan(o.float()).any() and bool(torch.isfinite(lse).all())
