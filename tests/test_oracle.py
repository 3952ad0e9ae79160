"""Pins for the FP64 oracle: checks against what the pages and mathematics fix.

No GPU.  Each pin compares the oracle with something other than itself: a
hand-derived closed form (tests/golden), torch's library attention and
logsumexp in float64, exact special cases (one visible key, q = 0, scale = 0,
rows with no visible key), structural identities (GQA equals MHA with
repeat_interleaved K/V, paged equals dense after scattering the cache through a
random block table, chunked prefill equals full prefill, row independence) and
invariants (convex hull, translation of V).  The optional terms are pinned the
same way: a zero left window leaves one key (exact value), a window equals the
plain definition over the sliced keys, softcap has closed forms for two keys
(tanh 40 = 1; 2 tanh(ln(3)/2) = 1) and vanishes for a huge cap, sinks obey the
denominator identity O_s = O / (1 + exp(s - LSE)), and paged equals dense with
all three.  Packed variable-length calls are checked request by request
against torch's attention, against the BSHD batch for equal lengths, and the
packed-query paged call against the packed call on gathered keys and against
the [B, Sq] paged call.  The last test plants mistakes in copies of the oracle and checks
that the pins catch every one.
"""
import math
import os
import shutil
import subprocess

import mpmath
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from gqa_softmax_attention_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "two_keys_closed_form.txt")


# ----------------------------------------------------------------------------- helpers
def _rand_case(B, Hq, Hkv, Sq, Skv, D, seed, mask_p=None, sigma=1.0):
    d = W.dense_inputs(B, Hq, Hkv, Sq, Skv, D, sigma=sigma, seed=seed)
    mask = None
    if mask_p is not None:
        g = torch.Generator().manual_seed(1000 + seed)
        mask = torch.rand(B, Skv, generator=g) < mask_p
    return d["q"], d["k"], d["v"], mask


def _visible(B, Sq, Skv, causal, mask):
    """[B, Sq, Skv] bool: key j visible to query i (end-aligned causal, padding)."""
    vis = torch.ones(B, Sq, Skv, dtype=torch.bool)
    if causal:
        vis &= torch.tril(torch.ones(Sq, Skv, dtype=torch.bool), diagonal=Skv - Sq)[None]
    if mask is not None:
        vis &= mask[:, None, :].bool()
    return vis


def _sdpa_fp64(q, k, v, mask, causal, scale):
    """torch's library attention in float64 (BSHD in, BSHD out)."""
    qf, kf, vf = (t.double().transpose(1, 2) for t in (q, k, v))
    B, Sq, Skv = q.shape[0], q.shape[1], k.shape[1]
    allowed = _visible(B, Sq, Skv, causal, mask)[:, None]
    out = F.scaled_dot_product_attention(qf, kf, vf, attn_mask=allowed, scale=scale,
                                         enable_gqa=True)
    return out.transpose(1, 2)


def _golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(None, 1)
            if key == "shape":
                vals[key] = {kv.split("=")[0]: float(kv.split("=")[1]) for kv in rest.split()}
            else:
                vals[key] = [float(x) for x in rest.split()]
    return vals


# ----------------------------------------------------------------------------- pins
def pin_golden_closed_form():
    g = _golden()
    s = {k: int(v) for k, v in g["shape"].items() if k != "scale"}
    B, Sq, Skv, Hq, Hkv, D = s["B"], s["Sq"], s["Skv"], s["Hq"], s["Hkv"], s["D"]
    q = torch.tensor(g["q"], dtype=torch.float64).view(B, Sq, Hq, D)
    k = torch.tensor(g["k"], dtype=torch.float64).view(B, Skv, Hkv, D)
    v = torch.tensor(g["v"], dtype=torch.float64).view(B, Skv, Hkv, D)
    o, lse = oracle.attn_dense(q, k, v, causal=True, scale=g["shape"]["scale"])
    assert torch.allclose(o.flatten(), torch.tensor(g["o"], dtype=torch.float64), atol=1e-15, rtol=0)
    assert torch.allclose(lse.flatten(), torch.tensor(g["lse"], dtype=torch.float64), atol=1e-15, rtol=0)
    mask = torch.tensor([[1, 0]], dtype=torch.bool)
    o, lse = oracle.attn_dense(q, k, v, key_padding_mask=mask, causal=False, scale=1.0)
    assert torch.equal(o.flatten(), torch.tensor(g["masked_o"], dtype=torch.float64))
    assert torch.equal(lse.flatten(), torch.tensor(g["masked_lse"], dtype=torch.float64))


SDPA_CASES = [
    # B, Hq, Hkv, Sq, Skv, D, causal, mask_p, scale
    (1, 4, 2, 8, 8, 8, True, None, None),
    (2, 4, 1, 5, 9, 4, True, 0.7, 0.37),
    (2, 6, 3, 7, 7, 16, False, 0.5, None),
    (1, 2, 2, 3, 11, 8, True, None, 1.7),
    (2, 8, 2, 6, 13, 8, False, None, -0.25),
    (1, 4, 4, 9, 5, 8, True, 0.8, None),      # Sq > Skv: leading rows see nothing
]


def pin_matches_torch_sdpa():
    for n, (B, Hq, Hkv, Sq, Skv, D, causal, mask_p, scale) in enumerate(SDPA_CASES):
        q, k, v, mask = _rand_case(B, Hq, Hkv, Sq, Skv, D, seed=n, mask_p=mask_p)
        o, lse = oracle.attn_dense(q, k, v, key_padding_mask=mask, causal=causal, scale=scale)
        ref = _sdpa_fp64(q, k, v, mask, causal, scale if scale is not None else 1 / math.sqrt(D))
        nonempty = _visible(B, Sq, Skv, causal, mask).any(-1)          # [B, Sq]
        rows = nonempty[:, :, None].expand(B, Sq, Hq)
        assert rows.any()
        err = (o - ref).abs()[rows].max().item()
        assert err < 1e-12, (n, err)


def pin_lse_matches_torch_logsumexp():
    for n, (B, Hq, Hkv, Sq, Skv, D, causal, mask_p, scale) in enumerate(SDPA_CASES):
        q, k, v, mask = _rand_case(B, Hq, Hkv, Sq, Skv, D, seed=n, mask_p=mask_p)
        sc = scale if scale is not None else 1 / math.sqrt(D)
        _, lse = oracle.attn_dense(q, k, v, key_padding_mask=mask, causal=causal, scale=scale)
        g = Hq // Hkv
        kk = k.double().repeat_interleave(g, dim=2)
        z = torch.einsum("bihd,bjhd->bhij", q.double(), kk) * sc
        vis = _visible(B, Sq, Skv, causal, mask)[:, None]
        z = z.masked_fill(~vis, float("-inf"))
        ref = torch.logsumexp(z, dim=-1).permute(0, 2, 1)              # [B, Sq, Hq]
        fin = torch.isfinite(ref)
        assert torch.equal(torch.isinf(lse), ~fin)
        assert (lse[fin] - ref[fin]).abs().max().item() < 1e-12


def pin_single_visible_key_exact():
    # causal, Sq == Skv: row 0 sees key 0 only -> O = V[0] exactly, LSE = scale <q0, k0>
    q, k, v, _ = _rand_case(2, 4, 2, 6, 6, 8, seed=7)
    scale = 0.3
    o, lse = oracle.attn_dense(q, k, v, causal=True, scale=scale)
    for b in range(2):
        for h in range(4):
            r = h // 2
            assert torch.equal(o[b, 0, h], v[b, 0, r].double())
            dot = math.fsum(float(a) * float(c) for a, c in zip(q[b, 0, h].double(), k[b, 0, r].double()))
            assert abs(lse[b, 0, h].item() - scale * dot) <= 1e-15 * max(1.0, abs(scale * dot))
    # a padding mask with exactly one kept key, no causal mask
    mask = torch.zeros(2, 6, dtype=torch.bool)
    mask[0, 3] = True
    mask[1, 5] = True
    o, lse = oracle.attn_dense(q, k, v, key_padding_mask=mask, causal=False)
    for b, j in ((0, 3), (1, 5)):
        for i in range(6):
            for h in range(4):
                assert torch.equal(o[b, i, h], v[b, j, h // 2].double())


def pin_zero_query_is_mean_of_visible_values():
    q, k, v, mask = _rand_case(2, 4, 2, 5, 9, 8, seed=11, mask_p=0.6)
    qz = torch.zeros_like(q)
    for qq, scale in ((qz, None), (q, 0.0)):
        o, lse = oracle.attn_dense(qq, k, v, key_padding_mask=mask, causal=True, scale=scale)
        vis = _visible(2, 5, 9, True, mask)
        for b in range(2):
            for i in range(5):
                js = torch.nonzero(vis[b, i]).flatten()
                for h in range(4):
                    if len(js) == 0:
                        assert torch.equal(o[b, i, h], torch.zeros(8, dtype=torch.float64))
                        assert lse[b, i, h].item() == float("-inf")
                        continue
                    vals = v[b, js, h // 2].double()
                    mean = torch.tensor([math.fsum(vals[:, d].tolist()) / len(js) for d in range(8)],
                                        dtype=torch.float64)
                    assert (o[b, i, h] - mean).abs().max().item() < 1e-15
                    assert lse[b, i, h].item() == math.log(len(js))


def pin_gqa_equals_repeat_interleave_mha():
    q, k, v, mask = _rand_case(2, 8, 2, 7, 10, 8, seed=3, mask_p=0.8)
    o, lse = oracle.attn_dense(q, k, v, key_padding_mask=mask, causal=True)
    km, vm = k.repeat_interleave(4, dim=2), v.repeat_interleave(4, dim=2)
    o2, lse2 = oracle.attn_dense(q, km, vm, key_padding_mask=mask, causal=True)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def _scatter_to_pages(k, v, lengths, page_size, seed, spare=3):
    """Lay dense [B, Skv, Hkv, D] K/V into a shuffled page pool (the inverse of a gather)."""
    B, Skv, Hkv, D = k.shape
    npages = [(int(L) + page_size - 1) // page_size for L in lengths]
    pool = sum(npages) + spare
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(pool, generator=g)
    max_pages = max(1, (Skv + page_size - 1) // page_size)
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    kc = torch.full((pool, page_size, Hkv, D), float("nan"), dtype=k.dtype)
    vc = torch.full((pool, page_size, Hkv, D), float("nan"), dtype=v.dtype)
    off = 0
    for b in range(B):
        for lp in range(npages[b]):
            phys = int(perm[off + lp])
            table[b, lp] = phys
            n = min(page_size, int(lengths[b]) - lp * page_size)
            kc[phys, :n] = k[b, lp * page_size: lp * page_size + n]
            vc[phys, :n] = v[b, lp * page_size: lp * page_size + n]
        off += npages[b]
    return kc, vc, table


def pin_paged_equals_dense():
    for n, (B, Sq, Hq, Hkv, D, ps) in enumerate(((3, 1, 4, 2, 8, 4), (2, 3, 6, 2, 8, 1),
                                                  (4, 2, 4, 4, 16, 16), (2, 4, 12, 1, 8, 3))):
        Skv = 21
        q, k, v, _ = _rand_case(B, Hq, Hkv, Sq, Skv, D, seed=20 + n)
        lengths = [Skv - 3 * b for b in range(B)]
        lengths[-1] = 0 if n == 0 else lengths[-1]             # an empty request
        kc, vc, table = _scatter_to_pages(k, v, lengths, ps, seed=50 + n)
        sl = torch.tensor(lengths, dtype=torch.int32)
        o, lse = oracle.attn_paged(q, kc, vc, sl, table, causal=True)
        for b in range(B):
            L = lengths[b]
            od, ld = oracle.attn_dense(q[b:b + 1], k[b:b + 1, :L], v[b:b + 1, :L], causal=True)
            assert torch.equal(o[b:b + 1], od) and torch.equal(lse[b:b + 1], ld)


def pin_rows_without_visible_keys():
    # causal with Sq > Skv: the first Sq - Skv rows see nothing
    q, k, v, _ = _rand_case(2, 4, 2, 9, 4, 8, seed=5)
    o, lse = oracle.attn_dense(q, k, v, causal=True)
    assert torch.equal(o[:, :5], torch.zeros_like(o[:, :5]))
    assert bool(torch.all(lse[:, :5] == float("-inf")))
    assert bool(torch.all(torch.isfinite(lse[:, 5:])))
    # Skv = 0
    o, lse = oracle.attn_dense(q, k[:, :0], v[:, :0], causal=False)
    assert torch.equal(o, torch.zeros_like(o)) and bool(torch.all(lse == float("-inf")))
    # a batch whose mask removes every key
    mask = torch.ones(2, 4, dtype=torch.bool)
    mask[1] = False
    o, lse = oracle.attn_dense(q, k, v, key_padding_mask=mask, causal=False)
    assert torch.equal(o[1], torch.zeros_like(o[1])) and bool(torch.all(lse[1] == float("-inf")))
    assert bool(torch.all(torch.isfinite(lse[0])))


def pin_invariants():
    q, k, v, mask = _rand_case(2, 4, 2, 6, 12, 8, seed=9, mask_p=0.7)
    o, lse = oracle.attn_dense(q, k, v, key_padding_mask=mask, causal=True)
    vis = _visible(2, 6, 12, True, mask)
    # convex hull of the visible value rows, per coordinate
    for b in range(2):
        for i in range(6):
            js = torch.nonzero(vis[b, i]).flatten()
            for h in range(4):
                if len(js) == 0:
                    continue
                vals = v[b, js, h // 2].double()
                assert bool(torch.all(o[b, i, h] >= vals.min(0).values - 1e-15))
                assert bool(torch.all(o[b, i, h] <= vals.max(0).values + 1e-15))
    # all value rows equal -> output is that row; weights sum to one
    vc = v[:, :1].expand_as(v).contiguous()
    o1, _ = oracle.attn_dense(q, k, vc, key_padding_mask=mask, causal=True)
    nonempty = vis.any(-1)
    for b in range(2):
        for i in range(6):
            if nonempty[b, i]:
                for h in range(4):
                    assert (o1[b, i, h] - vc[b, 0, h // 2].double()).abs().max().item() < 1e-15
    # translating every value row by c translates the output by c
    c = torch.linspace(-3, 3, 8, dtype=torch.float64)
    o2, lse2 = oracle.attn_dense(q.double(), k.double(), v.double() + c, key_padding_mask=mask,
                                 causal=True)
    rows = nonempty[:, :, None].expand(2, 6, 4)
    assert (o2 - c - o)[rows].abs().max().item() < 1e-13
    assert torch.equal(lse2, lse)


def pin_chunked_prefill_and_row_independence():
    q, k, v, _ = _rand_case(2, 4, 2, 16, 16, 8, seed=13)
    o, lse = oracle.attn_dense(q, k, v, causal=True)
    # chunk [c0, c1): Sq = c1 - c0 queries against the first c1 keys
    for c0, c1 in ((0, 5), (5, 11), (11, 16)):
        oc, lc = oracle.attn_dense(q[:, c0:c1], k[:, :c1], v[:, :c1], causal=True)
        assert torch.equal(oc, o[:, c0:c1]) and torch.equal(lc, lse[:, c0:c1])
    # a batch slice reproduces its rows exactly
    ob, lb = oracle.attn_dense(q[1:], k[1:], v[1:], causal=True)
    assert torch.equal(ob, o[1:]) and torch.equal(lb, lse[1:])
    # listed rows reproduce the full computation exactly
    rows = [(0, 0, 0), (1, 15, 3), (0, 7, 2), (1, 3, 1)]
    orow, lrow = oracle.attn_dense_rows(q, k, v, rows, causal=True)
    for n, (b, i, h) in enumerate(rows):
        assert torch.equal(orow[n], o[b, i, h]) and lrow[n].item() == lse[b, i, h].item()


def pin_noncausal_key_permutation():
    q, k, v, mask = _rand_case(1, 4, 2, 5, 10, 8, seed=17, mask_p=0.6)
    o, lse = oracle.attn_dense(q, k, v, key_padding_mask=mask, causal=False)
    perm = torch.randperm(10, generator=torch.Generator().manual_seed(4))
    o2, lse2 = oracle.attn_dense(q, k[:, perm], v[:, perm], key_padding_mask=mask[:, perm],
                                 causal=False)
    assert (o - o2).abs().max().item() < 1e-14
    assert (lse - lse2).abs().max().item() < 1e-14


def pin_high_precision_rows():
    """A few rows recomputed with 40-digit arithmetic (mpmath)."""
    q, k, v, mask = _rand_case(1, 4, 2, 6, 9, 8, seed=23, mask_p=0.7)
    scale = 1 / math.sqrt(8)
    o, lse = oracle.attn_dense(q, k, v, key_padding_mask=mask, causal=True)
    vis = _visible(1, 6, 9, True, mask)
    mpmath.mp.dps = 40
    for i, h in ((5, 0), (4, 3), (2, 1)):
        js = torch.nonzero(vis[0, i]).flatten().tolist()
        if not js:
            continue
        r = h // 2
        z = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(float(a)) * mpmath.mpf(float(b))
                                             for a, b in zip(q[0, i, h], k[0, j, r])) for j in js]
        den = mpmath.fsum(mpmath.e ** zj for zj in z)
        for d in range(8):
            num = mpmath.fsum(mpmath.e ** zj * mpmath.mpf(float(v[0, j, r, d])) for zj, j in zip(z, js))
            assert abs(float(num / den) - o[0, i, h, d].item()) < 1e-14
        assert abs(float(mpmath.log(den)) - lse[0, i, h].item()) < 1e-14


# ----------------------------------------------------------------------------- optional terms
# TileOPs "Attention Operators", GQADenseFwdOp stages 5 and 6 (window, softcap)
# and GQAPagedFwdOp's sinks.
def pin_window_single_key_exact():
    # causal with window_left = 0: row i sees key p_i only -> O = V[p_i] exactly,
    # LSE = scale <q_i, k_{p_i}>; the same with a cap (one key takes all the weight)
    q, k, v, _ = _rand_case(2, 4, 2, 5, 9, 8, seed=21)
    scale = 0.25
    for cap in (0.0, 0.3):
        o, lse = oracle.attn_dense(q, k, v, causal=True, scale=scale, window_left=0, softcap=cap)
        for b in range(2):
            for i in range(5):
                p = i + 9 - 5
                for h in range(4):
                    r = h // 2
                    assert torch.equal(o[b, i, h], v[b, p, r].double())
                    if cap == 0.0:
                        dot = math.fsum(float(a) * float(c) for a, c in zip(q[b, i, h].double(),
                                                                           k[b, p, r].double()))
                        assert abs(lse[b, i, h].item() - scale * dot) <= 1e-15 * max(1.0, abs(scale * dot))


def pin_window_equals_key_slice():
    # a window only removes keys: row i equals the plain non-causal definition over
    # keys [max(0, p_i - wL), min(Skv - 1, p_i (causal), p_i + wR)] alone
    B, Hq, Hkv, Sq, Skv, D = 1, 4, 2, 6, 14, 8
    q, k, v, mask = _rand_case(B, Hq, Hkv, Sq, Skv, D, seed=22, mask_p=0.8)
    for causal, wl, wr in ((True, 3, -1), (False, 2, 4), (False, 0, 0), (True, 20, -1), (False, -1, 1)):
        o, lse = oracle.attn_dense(q, k, v, key_padding_mask=mask, causal=causal, window_left=wl,
                                   window_right=wr)
        for i in range(Sq):
            p = i + Skv - Sq
            lo = 0 if wl < 0 else max(0, p - wl)
            hi = Skv - 1
            if causal:
                hi = min(hi, p)
            if wr >= 0:
                hi = min(hi, p + wr)
            if lo > hi or not bool(mask[0, lo:hi + 1].any()):
                assert torch.equal(o[0, i], torch.zeros(Hq, D, dtype=torch.float64))
                assert bool(torch.all(lse[0, i] == float("-inf")))
                continue
            ro, rl = oracle.attn_dense(q[:, i:i + 1], k[:, lo:hi + 1], v[:, lo:hi + 1],
                                       key_padding_mask=mask[:, lo:hi + 1], causal=False)
            assert (o[0, i] - ro[0, 0]).abs().max().item() < 1e-13
            assert (lse[0, i] - rl[0, 0]).abs().max().item() < 1e-13


def pin_softcap_closed_forms():
    # two visible keys, scaled scores z = (40, 0) and cap 1: logits (tanh 40 = 1, 0), so
    # the weights are e/(e+1), 1/(e+1) and LSE = log(e + 1); scores (ln 3, 0) and cap 2
    # give logits (2 tanh(ln(3)/2) = 1, 0): the same weights
    D = 4
    v = torch.tensor([[1.0, -2.0, 0.5, 3.0], [-1.0, 4.0, 2.0, 0.0]], dtype=torch.float64).view(1, 2, 1, D)
    w0 = math.e / (math.e + 1.0)
    want = w0 * v[0, 0, 0] + (1.0 - w0) * v[0, 1, 0]
    for z0, cap in ((40.0, 1.0), (math.log(3.0), 2.0)):
        q = torch.zeros(1, 1, 1, D, dtype=torch.float64)
        q[0, 0, 0, 0] = z0
        k = torch.zeros(1, 2, 1, D, dtype=torch.float64)
        k[0, 0, 0, 0] = 1.0
        o, lse = oracle.attn_dense(q, k, v, causal=False, scale=1.0, softcap=cap)
        assert (o[0, 0, 0] - want).abs().max().item() < 1e-14
        assert abs(lse[0, 0, 0].item() - math.log(math.e + 1.0)) < 1e-14


def pin_softcap_large_cap_limit():
    # c tanh(z / c) = z - z^3 / (3 c^2) + ...: a cap of 1e9 leaves the result unchanged
    q, k, v, mask = _rand_case(2, 4, 2, 5, 11, 8, seed=23, mask_p=0.7)
    o0, l0 = oracle.attn_dense(q, k, v, key_padding_mask=mask, causal=True)
    o1, l1 = oracle.attn_dense(q, k, v, key_padding_mask=mask, causal=True, softcap=1e9)
    assert (o0 - o1).abs().max().item() < 1e-12
    fin = torch.isfinite(l0)
    assert torch.equal(fin, torch.isfinite(l1))
    assert (l0[fin] - l1[fin]).abs().max().item() < 1e-12


def pin_sinks_identity():
    # a sink adds exp(s_h) to the denominator only: O_s = O exp(LSE) / (exp(LSE) + exp(s)),
    # LSE_s = log(exp(LSE) + exp(s)); s = -inf changes nothing, s = +inf zeroes the
    # output (LSE +inf); a row with no visible key stays zero with LSE -inf
    q, k, v, mask = _rand_case(2, 4, 2, 5, 7, 8, seed=24, mask_p=0.6)
    o0, l0 = oracle.attn_dense(q, k, v, key_padding_mask=mask, causal=True)
    inf = float("inf")
    sinks = torch.tensor([0.3, -1.5, 4.0, -inf], dtype=torch.float64)
    o1, l1 = oracle.attn_dense(q, k, v, key_padding_mask=mask, causal=True, sinks=sinks)
    for b in range(2):
        for i in range(5):
            for h in range(4):
                base, s = l0[b, i, h].item(), sinks[h].item()
                if base == -inf:
                    assert torch.equal(o1[b, i, h], torch.zeros(8, dtype=torch.float64))
                    assert l1[b, i, h].item() == -inf
                    continue
                frac = 1.0 / (1.0 + math.exp(s - base)) if s != -inf else 1.0
                assert (o1[b, i, h] - o0[b, i, h] * frac).abs().max().item() < 1e-13
                want = base if s == -inf else max(base, s) + math.log1p(math.exp(-abs(base - s)))
                assert abs(l1[b, i, h].item() - want) < 1e-13
    o2, l2 = oracle.attn_dense(q, k, v, key_padding_mask=mask, causal=True,
                               sinks=torch.tensor([inf, 0.0, 0.0, 0.0], dtype=torch.float64))
    has = torch.isfinite(l0[:, :, 0])
    assert bool(torch.all(o2[:, :, 0] == 0.0))
    assert bool(torch.all(l2[:, :, 0][has] == inf)) and bool(torch.all(l2[:, :, 0][~has] == -inf))


def pin_options_paged_equals_dense():
    # the optional terms act on the logical sequence: paged with window, cap and
    # sinks equals dense on the gathered cache
    q, k, v, _ = _rand_case(1, 4, 2, 3, 40, 8, seed=25)
    kc, vc, table = _scatter_to_pages(k, v, [40], 8, seed=5)
    sinks = torch.tensor([0.5, -0.5, 1.0, -2.0], dtype=torch.float64)
    od, ld = oracle.attn_dense(q, k, v, causal=True, window_left=9, softcap=5.0, sinks=sinks)
    op, lp = oracle.attn_paged(q, kc, vc, torch.tensor([40], dtype=torch.int32), table, causal=True,
                               window_left=9, softcap=5.0, sinks=sinks)
    assert (od - op).abs().max().item() < 1e-14
    assert (ld - lp).abs().max().item() < 1e-14


def pin_half_inputs_widen_exactly():
    # IEEE half inputs (the float16 calls of TileOPs GQAPagedFwdOp) widen to double
    # exactly: the oracle on float16 tensors equals the oracle on the same values
    # converted by torch to float64, bit for bit, including subnormals, signed
    # zeros and the largest finite half
    q, k, v, mask = _rand_case(2, 4, 2, 5, 9, 8, seed=26, mask_p=0.8)
    q16, k16, v16 = q.float().half(), k.float().half(), v.float().half()
    specials = torch.tensor([6.0e-8, -6.0e-8, 3.0e-6, -0.0, 0.0, 65504.0, -65504.0, 1.0 / 3.0],
                            dtype=torch.float16)
    v16[0, 0, 0, :] = specials
    k16[1, 2, 1, :] = specials * 1e-4
    for causal in (True, False):
        oh, lh = oracle.attn_dense(q16, k16, v16, key_padding_mask=mask, causal=causal)
        od, ld = oracle.attn_dense(q16.double(), k16.double(), v16.double(), key_padding_mask=mask, causal=causal)
        assert torch.equal(oh, od) and torch.equal(lh, ld)


def _pack(lengths, H, D, seed, stream):
    """A packed [sum(lengths), H, D] bf16 tensor and its [B + 1] offsets."""
    total = int(sum(lengths))
    x = W.randn_bf16((max(total, 1), H, D), seed=seed, stream=stream)[:total]
    cu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int32)
    return x, cu


def pin_varlen_matches_sdpa_per_request():
    # TileOPs GQAVarlenFwdOp: each request is attention over its own rows with
    # its own end-aligned causal mask; checked request by request against
    # torch's library attention (a request without queries, one with Sq > Skv)
    sq, skv = [3, 0, 5, 3, 1], [4, 2, 5, 1, 9]
    Hq, Hkv, D, scale = 4, 2, 8, 0.4
    q, cq = _pack(sq, Hq, D, seed=61, stream=0)
    k, ck = _pack(skv, Hkv, D, seed=61, stream=1)
    v, _ = _pack(skv, Hkv, D, seed=61, stream=2)
    o, lse = oracle.attn_varlen(q, k, v, cq, ck, causal=True, scale=scale)
    for b in range(len(sq)):
        qs, ks = int(cq[b]), int(ck[b])
        if sq[b] == 0:
            continue
        vis = _visible(1, sq[b], skv[b], True, None)[0].any(-1)          # rows with a visible key
        ref = _sdpa_fp64(q[None, qs:qs + sq[b]], k[None, ks:ks + skv[b]], v[None, ks:ks + skv[b]], None, True,
                         scale)[0]
        ob, lb = o[qs:qs + sq[b]], lse[qs:qs + sq[b]]
        assert torch.allclose(ob[vis], ref[vis], rtol=1e-12, atol=1e-12)
        assert torch.equal(ob[~vis], torch.zeros_like(ob[~vis])) and bool(torch.all(lb[~vis] == float("-inf")))
        assert bool(torch.all(torch.isfinite(lb[vis])))


def pin_varlen_equals_dense_batch():
    # equal lengths: the packed call is the BSHD batch, options included
    B, S, Skv, Hq, Hkv, D = 3, 6, 9, 6, 2, 8
    q, k, v, _ = _rand_case(B, Hq, Hkv, S, Skv, D, seed=62)
    cq = torch.arange(0, (B + 1) * S, S, dtype=torch.int32)
    ck = torch.arange(0, (B + 1) * Skv, Skv, dtype=torch.int32)
    sinks = torch.tensor([0.5, -1.0, float("-inf"), 2.0, 0.0, 1.0], dtype=torch.float64)
    for kw in ({}, dict(window_left=3, window_right=1, softcap=2.5, sinks=sinks)):
        o, lse = oracle.attn_varlen(q.reshape(B * S, Hq, D), k.reshape(B * Skv, Hkv, D), v.reshape(B * Skv, Hkv, D),
                                    cq, ck, causal=True, **kw)
        od, ld = oracle.attn_dense(q, k, v, causal=True, **kw)
        assert torch.equal(o, od.reshape(B * S, Hq, D)) and torch.equal(lse, ld.reshape(B * S, Hq))


def pin_paged_varlen_equals_gathered_varlen():
    # TileOPs GQAPagedFwdOp: packed queries over a paged cache whose lengths
    # include the query tokens equal the packed call on the gathered keys
    sq, L = [1, 0, 7, 1, 4], [13, 5, 7, 30, 11]
    Hq, Hkv, D, ps = 6, 2, 8, 4
    q, cq = _pack(sq, Hq, D, seed=63, stream=0)
    k, ck = _pack(L, Hkv, D, seed=63, stream=1)
    v, _ = _pack(L, Hkv, D, seed=63, stream=2)
    kd = torch.zeros(len(L), max(L), Hkv, D, dtype=k.dtype)
    vd = torch.zeros_like(kd)
    for b in range(len(L)):
        kd[b, :L[b]] = k[int(ck[b]):int(ck[b + 1])]
        vd[b, :L[b]] = v[int(ck[b]):int(ck[b + 1])]
    kc, vc, table = _scatter_to_pages(kd, vd, L, ps, seed=64)
    sl = torch.tensor(L, dtype=torch.int32)
    o, lse = oracle.attn_paged_varlen(q, kc, vc, cq, sl, table, causal=True)
    od, ld = oracle.attn_varlen(q, k, v, cq, ck, causal=True)
    assert torch.equal(o, od) and torch.equal(lse, ld)


def pin_paged_varlen_uniform_equals_paged():
    # every request with the same query count: the packed call is the [B, Sq] one
    B, Sq, Hq, Hkv, D, ps = 4, 2, 4, 1, 8, 3
    L = [2, 9, 17, 5]
    q, k, v, _ = _rand_case(B, Hq, Hkv, Sq, max(L), D, seed=65)
    kc, vc, table = _scatter_to_pages(k, v, L, ps, seed=66)
    sl = torch.tensor(L, dtype=torch.int32)
    cq = torch.arange(0, (B + 1) * Sq, Sq, dtype=torch.int32)
    o, lse = oracle.attn_paged_varlen(q.reshape(B * Sq, Hq, D), kc, vc, cq, sl, table, causal=True, softcap=3.0)
    op, lp = oracle.attn_paged(q, kc, vc, sl, table, causal=True, softcap=3.0)
    assert torch.equal(o, op.reshape(B * Sq, Hq, D)) and torch.equal(lse, lp.reshape(B * Sq, Hq))



# ----------------------------------------------------------------------------- float8_e4m3fn key/value caches
def _fp8_paged_case(B, Sq, Hq, Hkv, D, lengths, ps, seed):
    """Q (bf16), K/V as e4m3fn codes of N(0, 1) draws in a shuffled page pool
    (unused slots hold the NaN code), the table and the lengths."""
    q, k, v, _ = _rand_case(B, Hq, Hkv, Sq, max(lengths), D, seed=seed)
    k8 = k.float().to(torch.float8_e4m3fn).view(torch.uint8)
    v8 = v.float().to(torch.float8_e4m3fn).view(torch.uint8)
    npages = [(L + ps - 1) // ps for L in lengths]
    pool = sum(npages) + 2
    perm = torch.randperm(pool, generator=torch.Generator().manual_seed(seed + 500))
    table = torch.full((B, max(1, max(npages))), -1, dtype=torch.int32)
    kc = torch.full((pool, ps, Hkv, D), 0x7F, dtype=torch.uint8)
    vc = torch.full((pool, ps, Hkv, D), 0x7F, dtype=torch.uint8)
    off = 0
    for b in range(B):
        for lp in range(npages[b]):
            phys = int(perm[off + lp])
            table[b, lp] = phys
            n = min(ps, lengths[b] - lp * ps)
            kc[phys, :n] = k8[b, lp * ps: lp * ps + n]
            vc[phys, :n] = v8[b, lp * ps: lp * ps + n]
        off += npages[b]
    return q, kc, vc, table, torch.tensor(lengths, dtype=torch.int32)


def pin_e4m3_table_matches_library():
    # every e4m3fn code against torch's own float8_e4m3fn conversion (a library
    # routine): 0x7F and 0xFF are the only NaNs, everything else is exact
    codes = torch.arange(256, dtype=torch.uint8)
    mine = oracle.e4m3_decode(codes)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64)
    nan = torch.isnan(lib)
    assert torch.equal(torch.isnan(mine), nan) and int(nan.sum()) == 2
    assert torch.equal(mine[~nan], lib[~nan])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9 and mine[0x08] == 2.0 ** -6 and mine[0xB8] == -1.0


def pin_fp8kv_unit_scales_equals_paged():
    # unit scales: the FP8 call is the paged definition on the decoded values
    # (decoded here by torch), options included
    q, kc, vc, table, sl = _fp8_paged_case(3, 2, 6, 2, 16, [9, 0, 23], 4, seed=70)
    kd = kc.view(torch.float8_e4m3fn).to(torch.float64)
    vd = vc.view(torch.float8_e4m3fn).to(torch.float64)
    sinks = torch.tensor([0.5, -1.0, float("-inf"), 2.0, 0.0, 1.0], dtype=torch.float64)
    for kw in ({}, dict(window_left=5, window_right=0, softcap=4.0, sinks=sinks)):
        o, lse = oracle.attn_paged_fp8kv(q, kc, vc, None, None, sl, table, causal=True, **kw)
        op, lp = oracle.attn_paged(q.to(torch.float64), kd, vd, sl, table, causal=True, **kw)
        assert torch.equal(o, op) and torch.equal(lse, lp)


def pin_fp8kv_scale_roles():
    # k_scale[b, r] multiplies every score of KV head r in request b (the same
    # as that factor on the softmax scale), v_scale[b, r] multiplies its output
    # rows and leaves the log-sum-exp alone
    B, Sq, Hq, Hkv, D = 3, 2, 6, 3, 16
    q, kc, vc, table, sl = _fp8_paged_case(B, Sq, Hq, Hkv, D, [11, 17, 6], 4, seed=71)
    g = torch.Generator().manual_seed(72)
    ks = torch.rand(B, Hkv, generator=g, dtype=torch.float64) * 1.5 + 0.25
    vs = torch.rand(B, Hkv, generator=g, dtype=torch.float64) * 1.5 + 0.25
    scale = 0.3
    o, lse = oracle.attn_paged_fp8kv(q, kc, vc, ks, vs, sl, table, causal=True, scale=scale)
    gsz = Hq // Hkv
    for b in range(B):
        for r in range(Hkv):
            heads = slice(r * gsz, (r + 1) * gsz)
            o1, l1 = oracle.attn_paged_fp8kv(q, kc, vc, None, None, sl, table, causal=True,
                                             scale=scale * float(ks[b, r]))
            assert torch.allclose(o[b, :, heads], o1[b, :, heads] * float(vs[b, r]), rtol=1e-12, atol=1e-13)
            assert torch.allclose(lse[b, :, heads], l1[b, :, heads], rtol=1e-12, atol=1e-13)


PINS = [pin_golden_closed_form, pin_matches_torch_sdpa, pin_lse_matches_torch_logsumexp,
        pin_single_visible_key_exact, pin_zero_query_is_mean_of_visible_values,
        pin_gqa_equals_repeat_interleave_mha, pin_paged_equals_dense,
        pin_rows_without_visible_keys, pin_invariants, pin_chunked_prefill_and_row_independence,
        pin_noncausal_key_permutation, pin_high_precision_rows, pin_window_single_key_exact,
        pin_window_equals_key_slice, pin_softcap_closed_forms, pin_softcap_large_cap_limit,
        pin_sinks_identity, pin_options_paged_equals_dense, pin_half_inputs_widen_exactly,
        pin_varlen_matches_sdpa_per_request, pin_varlen_equals_dense_batch,
        pin_paged_varlen_equals_gathered_varlen, pin_paged_varlen_uniform_equals_paged,
        pin_e4m3_table_matches_library, pin_fp8kv_unit_scales_equals_paged, pin_fp8kv_scale_roles]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


def test_argument_errors():
    q, k, v, _ = _rand_case(1, 6, 4, 3, 3, 8, seed=1)     # Hq % Hkv != 0
    with pytest.raises(ValueError, match="divisible"):
        oracle.attn_dense(q, k, v)
    q, k, v, _ = _rand_case(1, 4, 2, 3, 8, 8, seed=1)
    kc, vc, table = _scatter_to_pages(k, v, [8], 4, seed=1)
    with pytest.raises(ValueError, match="length"):
        oracle.attn_paged(q, kc, vc, torch.tensor([9], dtype=torch.int32), table)
    bad = table.clone()
    bad[0, 0] = kc.shape[0]
    with pytest.raises(ValueError, match="block_table"):
        oracle.attn_paged(q, kc, vc, torch.tensor([8], dtype=torch.int32), bad)


def test_workload_generator_is_deterministic():
    a = W.dense_inputs(1, 2, 1, 5, 7, 8, seed=3, mask_lengths=(2, 7))
    b = W.dense_inputs(1, 2, 1, 5, 7, 8, seed=3, mask_lengths=(2, 7))
    assert torch.equal(a["q"], b["q"]) and torch.equal(a["key_padding_mask"], b["key_padding_mask"])
    big1 = W.randn_bf16((3 * W.CHUNK + 5,), seed=2, stream=1, threads=1)
    big2 = W.randn_bf16((3 * W.CHUNK + 5,), seed=2, stream=1, threads=4)
    assert torch.equal(big1, big2)
    p = W.paged_inputs(5, 2, 4, 2, 8, 16, lengths=(3, 70), seed=4)
    used = p["block_table"][p["block_table"] >= 0]
    assert len(torch.unique(used)) == len(used)                        # no page used twice
    assert int(used.max()) < p["num_pages"]
    for b in range(5):
        need = (int(p["real_seqlen_kv"][b]) + 15) // 16
        assert bool(torch.all(p["block_table"][b, :need] >= 0))
        assert bool(torch.all(p["block_table"][b, need:] == -1))


# ----------------------------------------------------------------------------- planted mistakes
MUTANTS = {
    "head_map_modulo": ("const int r = h / g;", "const int r = h % Hkv;"),
    "causal_top_left": ("const long p = (long)i + Skv - Sq;", "const long p = (long)i;"),
    "causal_off_by_one": ("(!causal || (long)j <= p)", "(!causal || (long)j < p)"),
    "window_left_off_by_one": ("(long)j >= p - opt->window_left", "(long)j > p - opt->window_left"),
    "window_right_ignored": ("(opt->window_right < 0 || (long)j <= p + opt->window_right)", "1"),
    "softcap_scale_dropped": ("opt->softcap * tanh(z[j] / opt->softcap)", "tanh(z[j] / opt->softcap)"),
    "sink_ignored": ("double Z = sink == -INFINITY ? 0.0 : exp(sink - M);", "double Z = 0.0;"),
    "sink_plus_inf_unhandled": ("if (sink == INFINITY) {", "if (0) {"),
    "half_exponent_bias": ("ldexp(1024.0 + m, e - 25)", "ldexp(1024.0 + m, e - 24)"),
    "half_subnormal_scale": ("ldexp((double)m, -24)", "ldexp((double)m, -23)"),
    "mask_ignored": ("mask[(size_t)b * Skv + j] != 0", "1"),
    "scale_dropped": ("z[j] = scale * dot;", "z[j] = dot;"),
    "lse_missing_log": ("*lse_out = M + log(Z);", "*lse_out = M + Z;"),
    "values_from_keys": ("w * load_elem(v, v_off + d, dtype)", "w * load_elem(k, v_off + d, dtype)"),
    "empty_row_lse_zero": ("*lse_out = -INFINITY;\n        return;", "*lse_out = 0;\n        return;"),
    "page_index_swapped": ("const long lp = t / page_size;", "const long lp = t % page_size;"),
    "weights_unnormalised": ("exp(z[j] - M) / Z;", "exp(z[j] - M);"),
    "query_row_transposed": ("(((size_t)b * Sq + i) * Hq + h)", "(((size_t)b * Hq + h) * Sq + i)"),
    "varlen_key_offset_ignored": ("(const char*)k + (size_t)ks * Hkv * D * es,", "(const char*)k,"),
    "varlen_output_offset_ignored": ("o + (size_t)qs * Hq * D, lse + (size_t)qs * Hq, 1, Hq, Hkv, sq,",
                                     "o, lse, 1, Hq, Hkv, sq,"),
    "paged_varlen_table_row_ignored": ("block_table + (size_t)b * max_pages, page_size, NULL,",
                                       "block_table, page_size, NULL,"),
    "paged_varlen_first_length": ("cache_seqlens + b,", "cache_seqlens,"),
    "e4m3_exponent_bias": ("ldexp(8.0 + m, e - 10)", "ldexp(8.0 + m, e - 9)"),
    "e4m3_subnormal_scale": ("ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    "e4m3_nan_missed": ("if (e == 15 && m == 7) mag = NAN;", "if (0) mag = NAN;"),
    "fp8_scales_swapped": ("e4m3_to_double(k_cache[src + e]) * ks;", "e4m3_to_double(k_cache[src + e]) * vs;"),
    "fp8_scale_request_ignored": ("k_scale[(size_t)b * Hkv + r]", "k_scale[r]"),
}


def _compile_mutant(tmp_path, name, old, new):
    src = open(oracle._build.SRC).read()
    assert src.count(old) == 1, name
    path = tmp_path / (name + ".c")
    path.write_text(src.replace(old, new))
    lib = tmp_path / ("lib" + name + ".so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", str(path), "-o", str(lib), "-lm"],
                   check=True, capture_output=True)
    return str(lib)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(tmp_path, name):
    old, new = MUTANTS[name]
    lib = _compile_mutant(tmp_path, name, old, new)
    caught = []
    with oracle.use_library(lib):
        for pin in PINS:
            try:
                pin()
            except (AssertionError, ValueError):
                caught.append(pin.__name__)
    assert caught, "no pin caught the planted mistake " + name
