"""The benchmark's multi-rank logic on CPU ranks (gloo, world size 2): the
max-over-ranks timing, the barrier and the whole-job aggregation that
`bench.py` uses when launched under torchrun.  No GPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.dist_env()
        assert (w, r, lr) == (world, rank, rank)
        bench.barrier(world)
        local = 0.010 + 0.005 * rank            # rank 1 is the slow one
        t = bench.max_over_ranks(local, world)
        out[rank] = t
        out[world + rank] = bench.job_value(0.004, t, world)
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Array("d", 2 * world)
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == pytest.approx(0.015) and out[1] == pytest.approx(0.015)
    # two replicas did twice the work of one in the slower rank's time
    assert out[2] == pytest.approx(100.0 * 2 * 0.004 / 0.015)
    assert out[2] == out[3]


def test_single_rank_defaults():
    assert bench.max_over_ranks(0.5, 1) == 0.5
    assert bench.job_value(1.0, 2.0, 1) == pytest.approx(50.0)


def test_visible_pairs_brute_force():
    g = torch.Generator().manual_seed(0)
    m = torch.rand(2, 37, generator=g) < 0.6
    for causal in (True, False):
        for Sq, Skv in ((37, 37), (10, 37), (40, 37)):
            bf = sum(1 for b in range(2) for i in range(Sq) for j in range(Skv)
                     if (not causal or j <= i + Skv - Sq) and m[b, j])
            assert bf == bench.visible_pairs(2, Sq, Skv, causal, m[:, :Skv])


def test_executed_work_counts_tiles_with_a_visible_pair():
    """Brute force over 128 x 128 tiles: a tile counts when any (row, key) in
    it is visible (causal, end-aligned, and the padding mask)."""
    torch.manual_seed(3)
    for B, Sq, Skv, causal in [(2, 200, 300, True), (1, 128, 128, True), (2, 130, 257, False), (1, 64, 400, True),
                               (1, 300, 200, True)]:
        mask = torch.rand(B, Skv) < 0.3
        mask[0, 128:256] = False                       # a whole key tile masked out
        d = dict(config=dict(B=B, Sq=Sq, Skv=Skv, D=64, Hq=3, causal=causal), key_padding_mask=mask)
        tiles = 0
        for b in range(B):
            for q0 in range(0, Sq, 128):
                for k0 in range(0, Skv, 128):
                    rows = torch.arange(q0, min(q0 + 128, Sq))[:, None]
                    keys = torch.arange(k0, min(k0 + 128, Skv))[None, :]
                    vis = mask[b, k0:k0 + 128][None, :].expand(rows.shape[0], -1).clone()
                    if causal:
                        vis &= keys <= rows + Skv - Sq
                    tiles += int(bool(vis.any()))
        assert bench.executed_work(d) == 4.0 * 128 * 128 * 64 * 3 * tiles


def test_decode_bytes_count_the_element_size():
    from gqa_softmax_attention_gb300 import workloads as W
    for kind, gen, elem in (("paged", W.paged_inputs, 2), ("paged_fp8", W.paged_fp8_inputs, 1)):
        cfg = dict(kind=kind, B=3, Sq=1, Hq=8, Hkv=2, D=128, page_size=16, lengths=[5, 0, 70])
        d = gen(**cfg)
        d["config"] = cfg
        assert bench.decode_bytes(d) == (5 + 0 + 70) * 2 * 2 * 128 * elem


def test_fp8_inputs_are_e4m3_with_scales_in_range():
    from gqa_softmax_attention_gb300 import workloads as W
    d = W.paged_fp8_inputs(4, 2, 8, 2, 128, 16, lengths=(1, 300), seed=3, scale_range=(0.25, 1.0))
    assert d["k_cache"].dtype == torch.float8_e4m3fn and d["v_cache"].dtype == torch.float8_e4m3fn
    for n in ("k_scale", "v_scale"):
        s = d[n]
        assert s.shape == (4, 2) and s.dtype == torch.float32
        assert bool(((s >= 0.25) & (s < 1.0)).all())
    codes = d["k_cache"].view(torch.uint8)
    assert not bool(((codes & 0x7F) == 0x7F).any())          # no NaN code anywhere
    # the same seed draws the same bytes and scales
    e = W.paged_fp8_inputs(4, 2, 8, 2, 128, 16, lengths=(1, 300), seed=3, scale_range=(0.25, 1.0))
    assert torch.equal(codes, e["k_cache"].view(torch.uint8)) and torch.equal(d["v_scale"], e["v_scale"])


def _part(kind, gen, cfg):
    d = gen(**cfg)
    d["config"] = dict(cfg, kind=kind)
    return bench.Part("probe", d)


def test_oracle_sample_of_a_dense_part_counts_its_rows_flops():
    from gqa_softmax_attention_gb300 import workloads as W
    cfg = dict(B=2, Hq=4, Hkv=2, Sq=40, Skv=70, D=64, causal=True, sigma=1.0, mask_lengths=(30, 70), seed=5)
    p = _part("dense", W.dense_inputs, cfg)
    unit, rows, flops, nbytes = bench._draw_sample(p, 0.25, torch.Generator().manual_seed(0))
    assert unit == "rows" and len(rows) == 80 and nbytes == 0.0
    m = p.data["key_padding_mask"]
    pairs = sum(1 for b, i, _h in rows for j in range(70) if j <= i + 70 - 40 and m[b, j])
    assert flops == 4.0 * 64 * pairs
    assert bench._run_sample(p, unit, rows) >= 0.0


def test_decode_sample_units_reproduce_the_full_call():
    # the compact call built from sampled (request, query head) pairs gives the
    # oracle's own rows of the full paged call, bit for bit
    import oracle
    from gqa_softmax_attention_gb300 import workloads as W
    for kind, gen in (("paged", W.paged_inputs), ("paged_fp8", W.paged_fp8_inputs)):
        cfg = dict(B=4, Sq=3, Hq=6, Hkv=2, D=64, page_size=8, lengths=[19, 0, 2, 33], seed=7)
        if kind == "paged_fp8":
            cfg["scale_range"] = (0.25, 1.0)
        p = _part(kind, gen, cfg)
        d = p.data
        unit, units, flops, nbytes = bench._draw_sample(p, 0.5, torch.Generator().manual_seed(1))
        assert flops == 0.0 and len(units) >= 1
        elem = 1 if kind == "paged_fp8" else 2
        want = sum(d["real_seqlen_kv"][b].item() * 2 * 64 * elem / 3 for b, _h in units)
        assert nbytes == pytest.approx(want)
        u = bench._decode_units(p, units)
        if kind == "paged":
            full = oracle.attn_paged(d["q"], d["k_cache"], d["v_cache"], d["real_seqlen_kv"], d["block_table"])
            part = oracle.attn_paged(u["q"], u["k_cache"], u["v_cache"], u["real_seqlen_kv"], u["block_table"])
        else:
            full = oracle.attn_paged_fp8kv(d["q"], d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"],
                                           d["real_seqlen_kv"], d["block_table"])
            part = oracle.attn_paged_fp8kv(u["q"], u["k_cache"], u["v_cache"], u["k_scale"], u["v_scale"],
                                           u["real_seqlen_kv"], u["block_table"])
        for i, (b, h) in enumerate(units):
            assert torch.equal(part[0][i, :, 0], full[0][b, :, h])
            assert torch.equal(part[1][i, :, 0], full[1][b, :, h])


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` runs the oracle on the host cores and prints
    one JSON line with the contract's keys (small workload, three steps)."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_dense", "--steps", "3",
                        "--warmup", "3"], cwd=root, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"]
