"""float16 inputs on the GPU against the FP64 oracle.

TileOPs "Attention Operators" serves Q and the cache in "a float16 or bfloat16
dtype" (GQAPagedFwdOp); here every kernel takes either, selected per call
(gqa_options.dtype), with FP32 products and sums and P rounded to the call's
type before P V.  The oracle widens the same float16 bits exactly.
"""
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


def half(t):
    return t.float().half()


DENSE = [
    # B, Hq, Hkv, Sq, Skv, D, causal, window_left
    (1, 4, 2, 128, 128, 64, True, -1),
    (2, 8, 2, 300, 700, 128, True, -1),
    (2, 4, 1, 190, 400, 128, False, -1),
    (1, 8, 2, 257, 513, 128, True, 100),
]


@pytest.mark.parametrize("case", DENSE, ids=[str(c) for c in DENSE])
def test_dense_fp16(g, case):
    B, Hq, Hkv, Sq, Skv, D, causal, wl = case
    d = W.dense_inputs(B, Hq, Hkv, Sq, Skv, D, seed=Sq + Skv + 1)
    q, k, v = half(d["q"]), half(d["k"]), half(d["v"])
    o, lse = g.attention(q.cuda(), k.cuda(), v.cuda(), causal=causal, window_left=wl)
    torch.cuda.synchronize()
    assert o.dtype == torch.float16
    ro, rl = oracle.attn_dense(q, k, v, causal=causal, window_left=wl)
    compare(o, lse, ro, rl, str(case))


PAGED = [
    # B, Sq, Hq, Hkv, D, page_size, lengths                  (rows per KV head -> path)
    (5, 1, 8, 2, 128, 16, [1, 0, 300, 17, 2000]),             # split kernel, TMA pages
    (3, 2, 32, 4, 128, 3, [50, 401, 1000]),                   # split kernel, gathered pages
    (4, 4, 24, 2, 256, 16, [3, 700, 129, 3000]),              # tensor-core kernel
    (2, 4, 32, 1, 128, 64, [129, 5000]),                      # tensor-core kernel, 128 rows
]


@pytest.mark.parametrize("case", PAGED, ids=[str(c[:6]) for c in PAGED])
def test_paged_fp16(g, case):
    B, Sq, Hq, Hkv, D, ps, lengths = case
    p = W.paged_inputs(B, Sq, Hq, Hkv, D, ps, lengths=lengths, seed=sum(lengths) % 83)
    q, kc, vc = half(p["q"]), half(p["k_cache"]), half(p["v_cache"])
    o, lse = g.decode_paged(q.cuda(), kc.cuda(), vc.cuda(), p["real_seqlen_kv"].cuda(), p["block_table"].cuda())
    torch.cuda.synchronize()
    assert o.dtype == torch.float16
    ro, rl = oracle.attn_paged(q, kc, vc, p["real_seqlen_kv"], p["block_table"])
    compare(o, lse, ro, rl, str(case))


def test_mixed_dtypes_refused(g):
    d = W.dense_inputs(1, 4, 2, 64, 64, 64, seed=1)
    with pytest.raises(ValueError, match="dtype|float16|bfloat16"):
        g.attention(d["q"].cuda(), half(d["k"]).cuda(), d["v"].cuda())
