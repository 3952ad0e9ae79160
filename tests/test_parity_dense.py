"""Dense prefill on the GPU against the FP64 oracle (through the C ABI)."""
import pytest
import torch

import oracle
from gqa_softmax_attention_gb300 import workloads as W

from parity import compare, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gqa_softmax_attention_gb300 import build
    build.build()
    import gqa_softmax_attention_gb300 as m
    yield m
    m.gqa_device_error()          # no kernel wait may have timed out


def run(g, d, causal=True, scale=None, mask=None):
    dev = "cuda"
    q, k, v = d["q"].to(dev), d["k"].to(dev), d["v"].to(dev)
    m = mask.to(dev) if mask is not None else None
    o, lse = g.attention(q, k, v, causal=causal, scale=scale, key_padding_mask=m)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def random_mask(B, Skv, p, seed):
    gen = torch.Generator().manual_seed(seed)
    return torch.rand(B, Skv, generator=gen) < p


SMALL = [
    # B, Hq, Hkv, Sq, Skv, D, causal, mask, scale
    (1, 4, 2, 128, 128, 64, True, None, None),
    (2, 8, 2, 200, 200, 128, True, None, None),          # ragged tail, two query tiles
    (1, 4, 4, 300, 700, 64, True, None, None),           # chunked prefill shape, MHA
    (2, 6, 3, 257, 129, 128, True, None, None),          # Sq > Skv: leading rows empty
    (2, 4, 1, 130, 390, 128, False, 0.5, None),          # random padding, non-causal
    (2, 8, 2, 256, 384, 128, True, "prefix", None),      # prefix padding, one batch empty
    (1, 2, 1, 64, 1000, 64, False, "runs", None),        # long padded runs: tile skipping
    (1, 4, 2, 190, 190, 128, True, None, 0.0),           # scale 0: mean of visible values
    (2, 4, 2, 129, 260, 64, True, 0.8, 0.3),
    (1, 16, 2, 512, 512, 128, True, None, None),         # several tiles, g = 8
]


@pytest.mark.parametrize("case", SMALL, ids=[str(c[:7]) for c in SMALL])
def test_small_shapes(g, case):
    B, Hq, Hkv, Sq, Skv, D, causal, mk, scale = case
    d = W.dense_inputs(B, Hq, Hkv, Sq, Skv, D, seed=Sq + Skv)
    mask = None
    if mk == "prefix":
        mask = torch.arange(Skv)[None, :] < torch.tensor([[Skv // 3], [0]])
    elif mk == "runs":
        mask = torch.zeros(B, Skv, dtype=torch.bool)
        mask[:, 5:9] = True
        mask[:, 600:900] = True
    elif mk is not None:
        mask = random_mask(B, Skv, mk, seed=Sq)
    q0, k0, v0 = d["q"].clone(), d["k"].clone(), d["v"].clone()
    o, lse = run(g, d, causal, scale, mask)
    ro, rl = oracle.attn_dense(d["q"], d["k"], d["v"], key_padding_mask=mask, causal=causal, scale=scale)
    compare(o, lse, ro, rl, str(case))
    assert torch.equal(q0, d["q"]) and torch.equal(k0, d["k"]) and torch.equal(v0, d["v"])


def test_tiny_workload(g):
    d = W.make("tiny_dense")
    o, lse = run(g, d)
    ro, rl = oracle.attn_dense(d["q"], d["k"], d["v"], causal=True)
    compare(o, lse, ro, rl, "tiny_dense")


def test_single_visible_key_is_exact(g):
    # causal, Sq == Skv: row 0 sees key 0 only, so P = 1 exactly and O = V[0] bit for bit
    d = W.dense_inputs(2, 8, 2, 160, 160, 128, seed=5)
    o, lse = run(g, d, causal=True, scale=0.25)
    for b in range(2):
        for h in range(8):
            assert torch.equal(o[b, 0, h], d["v"][b, 0, h // 4])
            ref = 0.25 * float((d["q"][b, 0, h].double() * d["k"][b, 0, h // 4].double()).sum())
            assert abs(float(lse[b, 0, h]) - ref) < 1e-4


def test_empty_key_axis(g):
    d = W.dense_inputs(2, 4, 2, 33, 0, 64, seed=1)
    o, lse = run(g, d)
    assert bool(torch.all(o == 0)) and bool(torch.all(torch.isneginf(lse)))


def test_chunked_prefill_matches_full(g):
    d = W.dense_inputs(1, 8, 2, 640, 640, 128, seed=9)
    o, lse = run(g, d)
    for c0, c1 in ((0, 256), (256, 512), (512, 640)):
        part = dict(q=d["q"][:, c0:c1].contiguous(), k=d["k"][:, :c1].contiguous(), v=d["v"][:, :c1].contiguous())
        oc, lc = run(g, part)
        compare(oc, lc, o[:, c0:c1].double(), lse[:, c0:c1].double(), "chunk %d:%d" % (c0, c1))


def test_batch_rows_are_independent(g):
    d = W.dense_inputs(3, 4, 2, 200, 300, 64, seed=2)
    o, lse = run(g, d)
    part = dict(q=d["q"][1:2].contiguous(), k=d["k"][1:2].contiguous(), v=d["v"][1:2].contiguous())
    o1, l1 = run(g, part)
    assert torch.equal(o1, o[1:2]) and torch.equal(l1, lse[1:2])     # bitwise: same tiles, same order


def test_gqa_equals_repeated_kv(g):
    d = W.dense_inputs(1, 8, 2, 256, 256, 128, seed=4)
    o, lse = run(g, d)
    rep = dict(q=d["q"], k=d["k"].repeat_interleave(4, dim=2).contiguous(),
               v=d["v"].repeat_interleave(4, dim=2).contiguous())
    o2, l2 = run(g, rep)
    assert torch.equal(o, o2) and torch.equal(lse, l2)


@pytest.mark.parametrize("name", ["qwen3_8b_prefill", "long_chunked_prefill"])
def test_full_size_workload_sampled_rows(g, name):
    d = W.make(name)
    cfg = d["config"]
    o, lse = run(g, d, mask=d["key_padding_mask"])
    rows = sample_rows(cfg["B"], cfg["Sq"], cfg["Hq"], lengths=d["lengths"], extra=96)
    ro, rl = oracle.attn_dense_rows(d["q"], d["k"], d["v"], rows, key_padding_mask=d["key_padding_mask"],
                                    causal=True)
    idx = torch.tensor(rows)
    stats = compare(o[idx[:, 0], idx[:, 1], idx[:, 2]], lse[idx[:, 0], idx[:, 1], idx[:, 2]], ro, rl, name)
    assert stats["rows"] > 0
    # properties that hold for every row at any size: nothing is NaN, and since
    # every row of these workloads sees at least key 0, no LSE is -inf
    assert not torch.isnan(o.float()).any() and not torch.isnan(lse).any()
    assert bool(torch.isfinite(lse).all())
