#!/usr/bin/env python
"""Benchmark of the causal GQA attention forward hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  * dense prefill, Qwen3-8B-shaped: B=2, Sq=Skv=4096, Hq=32, Hkv=8, D=128,
    causal, key_padding_mask with per-batch valid lengths U[2048, 4096];
  * paged decode of the same geometry: B=64, Sq=1, ps=64, lengths
    U[1024, 16384], pages shuffled through block_table.
Inputs are resident in HBM before timing.  Work is counted algorithmically:
prefill FLOPs = 4 * D * Hq * (visible query/key pairs), decode bytes = the K
and V bytes of the real tokens (one byte per element for e4m3fn caches).  The reported value is the step's roofline
efficiency, 100 * (FLOPs / tensor peak + bytes / HBM peak) / step time, with
the measured peaks of this machine; per-kernel TFLOP/s and GB/s are reported
beside it.  Between timed steps a buffer twice the L2 size is overwritten so
every step starts with a cold L2.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload step|qwen3_8b_prefill|paged_decode|wide_group_decode|long_chunked_prefill|
                                   wide_group_prefill|varlen_prefill|mixed_serving_batch|paged_decode_fp8kv]
Prints exactly one JSON line (rank 0).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from gqa_softmax_attention_gb300 import workloads as W  # noqa: E402

METRIC = "prefill TFLOP/s and paged-decode HBM GB/s, as % of GB300 roofline"
UNIT = "% of roofline"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------------- work accounting
def visible_pairs(B, Sq, Skv, causal, mask):
    """Sum over batches and query rows of the number of visible keys."""
    i = torch.arange(Sq, dtype=torch.int64)
    lim = (i + Skv - Sq + 1).clamp(0, Skv) if causal else torch.full((Sq,), Skv, dtype=torch.int64)
    if mask is None:
        return int(lim.sum()) * B
    total = 0
    for b in range(B):
        c = torch.cat([torch.zeros(1, dtype=torch.int64), mask[b].to(torch.int64).cumsum(0)])
        total += int(c[lim].sum())
    return total


def prefill_work(d):
    c = d["config"]
    pairs = visible_pairs(c["B"], c["Sq"], c["Skv"], c["causal"], d["key_padding_mask"])
    return 4.0 * c["D"] * c["Hq"] * pairs, pairs


def decode_bytes(p):
    """K/V bytes of the real tokens: 2 bytes per element, 1 for e4m3fn caches."""
    c = p["config"]
    elem = 1 if c["kind"] == "paged_fp8" else 2
    return float(p["real_seqlen_kv"].to(torch.int64).sum()) * 2 * c["Hkv"] * c["D"] * elem


def packed_pairs(cu_q, kv_lens):
    """Visible (query, key) pairs of a packed causal call, one head: query i of
    request b sees min(L_b, i + L_b - Sq_b + 1) keys (end-aligned)."""
    total = 0
    for b in range(len(kv_lens)):
        sq, L = int(cu_q[b + 1] - cu_q[b]), int(kv_lens[b])
        i = torch.arange(sq, dtype=torch.int64)
        total += int((i + L - sq + 1).clamp(0, L).sum())
    return total


def packed_work(d):
    """(FLOPs, pairs per head, K/V bytes read once) of a packed call."""
    c = d["config"]
    if c["kind"] == "varlen":
        lens = (d["cu_seqlens_kv"][1:] - d["cu_seqlens_kv"][:-1]).tolist()
    else:
        lens = d["cache_seqlens"].tolist()
    pairs = packed_pairs(d["cu_seqlens_q"], lens)
    kv_bytes = float(sum(lens)) * 2 * c["Hkv"] * c["D"] * 2
    return 4.0 * c["D"] * c["Hq"] * pairs, pairs, kv_bytes


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return dict(hbm_gbs=float(pk["hbm_gbs"]), bf16_tflops=float(pk["bf16_tflops"]),
                    bf16_tflops_sustained=float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                    source="measured")
    return dict(FALLBACK, source="fallback")


# --------------------------------------------------------------------------- workload
# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the dominant
# kernel, taken once with ncu on the kernel as it stands: for the decode
# workloads as a ratio to the algorithmic K/V bytes (their captures ran at a
# reduced batch), for the prefill as bytes per launch of the same workload.
# A workload whose dominant kernel changed after its capture has no entry (its
# traffic is reported as null until it is captured again): qwen3_8b_prefill and
# long_chunked_prefill (prefill_kernel, epilogue store wait moved) and
# wide_group_decode (decode_tc_kernel, shared with the e4m3 route since).
TRAFFIC = {
    "paged_decode": ("ratio", (559.379712 + 6.031616) / 556.916736),
    "paged_decode_fp8kv": ("ratio", (279.805952 + 5.622016) / 278.458368),
    "wide_group_decode_fp8kv": ("ratio", (117.060352 + 3.536896) / 116.341760),
    "wide_group_prefill": ("bytes", (235.505152 + 160.755456) * 1e6),
    "mixed_serving_batch": ("bytes", (2583.485 + 24.447744) * 1e6),
    "varlen_prefill": ("bytes", (6572.479 + 507.1168) * 1e6),
}


def traffic_per_launch(part):
    t = TRAFFIC.get(part.name)
    if t is None:
        return None
    return t[1] * part.bytes if t[0] == "ratio" else t[1]


class Part:
    """One piece of the step: a dense prefill or a paged decode."""

    def __init__(self, name, data):
        self.name = name
        self.data = data
        self.kind = data["config"]["kind"]
        if self.kind == "dense":
            self.flops, self.pairs = prefill_work(data)
            self.bytes = 0.0
        elif self.kind == "varlen":
            self.flops, self.pairs, _ = packed_work(data)      # tensor-bound: FLOPs only
            self.bytes = 0.0
        elif self.kind == "paged_varlen":
            # prefill chunks and decode steps together: both terms count
            self.flops, self.pairs, self.bytes = packed_work(data)
        else:
            self.flops, self.pairs = 0.0, 0
            self.bytes = decode_bytes(data)

    def ideal_s(self, peaks):
        return self.flops / (peaks["bf16_tflops"] * 1e12) + self.bytes / (peaks["hbm_gbs"] * 1e9)

    def to_device(self, dev):
        d = self.data
        if self.kind in ("varlen", "paged_varlen"):
            import gqa_softmax_attention_gb300 as g
            c = d["config"]
            if self.kind == "varlen":
                names = ("q", "k", "v", "cu_seqlens_q", "cu_seqlens_kv")
            else:
                names = ("q", "k_cache", "v_cache", "cu_seqlens_q", "cache_seqlens", "block_table")
            self.dev = {n: d[n].to(dev) for n in names}
            tq = d["q"].shape[0]
            need = g.attn_varlen_workspace_size(len(d["cu_seqlens_q"]) - 1, tq, c["Hq"], c["Hkv"])
            self.dev["ws"] = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
            self.dev["o"] = torch.empty_like(self.dev["q"])
            self.dev["lse"] = torch.empty((tq, c["Hq"]), dtype=torch.float32, device=dev)
            return
        if self.kind == "dense":
            self.dev = dict(q=d["q"].to(dev), k=d["k"].to(dev), v=d["v"].to(dev),
                            m=d["key_padding_mask"].to(dev) if d["key_padding_mask"] is not None else None)
            c = d["config"]
            self.dev["o"] = torch.empty_like(self.dev["q"])
            self.dev["lse"] = torch.empty((c["B"], c["Sq"], c["Hq"]), dtype=torch.float32, device=dev)
        else:
            import gqa_softmax_attention_gb300 as g
            c = d["config"]
            self.dev = dict(q=d["q"].to(dev), kc=d["k_cache"].to(dev), vc=d["v_cache"].to(dev),
                            sl=d["real_seqlen_kv"].to(dev), bt=d["block_table"].to(dev))
            if self.kind == "paged_fp8":
                self.dev.update(ks=d["k_scale"].to(dev), vs=d["v_scale"].to(dev))
            need = g.attn_decode_paged_workspace_size(c["B"], c["Sq"], c["Hq"], c["Hkv"], c["D"], c["page_size"],
                                                      d["max_pages"])
            self.dev["ws"] = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
            self.dev["o"] = torch.empty_like(self.dev["q"])
            self.dev["lse"] = torch.empty((c["B"], c["Sq"], c["Hq"]), dtype=torch.float32, device=dev)

    def launches(self):
        return 1 if self.kind == "dense" else 2           # packed calls: plan + attention

    def run(self):
        import gqa_softmax_attention_gb300 as g
        x = self.dev
        if self.kind == "varlen":
            g.attn_fwd_varlen(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_kv"], causal=True,
                              out=x["o"], lse=x["lse"], workspace=x["ws"])
        elif self.kind == "paged_varlen":
            g.attn_fwd_paged(x["q"], x["k_cache"], x["v_cache"], x["cu_seqlens_q"], x["cache_seqlens"],
                             x["block_table"], causal=True, out=x["o"], lse=x["lse"], workspace=x["ws"])
        elif self.kind == "dense":
            g.attn_fwd_dense(x["q"], x["k"], x["v"], key_padding_mask=x["m"], causal=True, out=x["o"], lse=x["lse"])
        elif self.kind == "paged_fp8":
            g.attn_decode_paged_fp8kv(x["q"], x["kc"], x["vc"], x["ks"], x["vs"], x["sl"], x["bt"], causal=True,
                                      workspace=x["ws"], out=x["o"], lse=x["lse"])
        else:
            g.attn_decode_paged(x["q"], x["kc"], x["vc"], x["sl"], x["bt"], causal=True, workspace=x["ws"],
                                out=x["o"], lse=x["lse"])

    # host-resident copies for the end-to-end measurement
    def pin(self):
        d = self.data
        if self.kind == "varlen":
            names = [(n, d[n]) for n in ("q", "k", "v", "cu_seqlens_q", "cu_seqlens_kv")]
        elif self.kind == "paged_varlen":
            names = [(n, d[n]) for n in ("q", "k_cache", "v_cache", "cu_seqlens_q", "cache_seqlens", "block_table")]
        elif self.kind == "dense":
            names = [("q", d["q"]), ("k", d["k"]), ("v", d["v"])]
            if d["key_padding_mask"] is not None:
                names.append(("m", d["key_padding_mask"]))
        else:
            names = [("q", d["q"]), ("kc", d["k_cache"]), ("vc", d["v_cache"]), ("sl", d["real_seqlen_kv"]),
                     ("bt", d["block_table"])]
            if self.kind == "paged_fp8":
                names += [("ks", d["k_scale"]), ("vs", d["v_scale"])]
        self.host_in = [(n, t.contiguous().pin_memory()) for n, t in names]
        self.host_out = [("o", torch.empty(self.dev["o"].shape, dtype=self.dev["o"].dtype).pin_memory()),
                         ("lse", torch.empty(self.dev["lse"].shape, dtype=torch.float32).pin_memory())]

    def h2d(self):
        n = 0
        for name, t in self.host_in:
            self.dev[name].copy_(t, non_blocking=True)
            n += t.numel() * t.element_size()
        return n

    def d2h(self):
        n = 0
        for name, t in self.host_out:
            t.copy_(self.dev[name], non_blocking=True)
            n += t.numel() * t.element_size()
        return n


def make_parts(workload, batch=None):
    """The step's parts; `batch` shrinks a single named workload's B (for profiling captures)."""
    names = ["qwen3_8b_prefill", "paged_decode"] if workload == "step" else [workload]
    parts = []
    for n in names:
        if batch is None:
            parts.append(Part(n, W.make(n)))
            continue
        cfg = dict(W.WORKLOADS[n], B=batch)
        if cfg["kind"] not in ("dense", "paged", "paged_fp8"):
            raise SystemExit("--batch applies to the dense and paged-decode workloads")
        make_in = {"dense": W.dense_inputs, "paged": W.paged_inputs, "paged_fp8": W.paged_fp8_inputs}[cfg["kind"]]
        data = make_in(**cfg)
        data["config"] = cfg
        parts.append(Part(n, data))
    return parts


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.first = ""
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        self.cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "50"] + sel

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.first = self.proc.stdout.readline()   # wait for the first sample
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = [r.split(",") for r in (self.first + out).strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        reasons = set()
        for r in rows:
            for name, col in (("hw_slowdown", 5), ("hw_thermal_slowdown", 6), ("sw_thermal_slowdown", 7),
                              ("sw_power_cap", 8)):
                if r[col].strip().lower() == "active":
                    reasons.add(name)
        return dict(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=max(mx) if mx else None,
                    reasons=sorted(reasons), samples=len(rows))


# --------------------------------------------------------------------------- distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(ideal_s_per_rank, step_s_max, world):
    """Whole-job value: every rank ran the same step (replicas), so the job did
    `world` times the work of one rank in the slowest rank's time."""
    return 100.0 * world * ideal_s_per_rank / step_s_max


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------- our arm
def bench_ours(args, world, rank, local):
    import gqa_softmax_attention_gb300 as g
    from gqa_softmax_attention_gb300 import _lib
    _lib.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    parts = make_parts(args.workload, args.batch)
    for p in parts:
        p.to_device(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        flush.zero_()
        for p in parts:
            p.run()
    torch.cuda.synchronize(dev)
    g.gqa_device_error()

    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in parts]
          for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for s in range(args.steps):
        flush.zero_()                            # cold L2 for every step (outside the events)
        for j, p in enumerate(parts):
            ev[s][j][0].record(stream)
            p.run()
            ev[s][j][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    g.gqa_device_error()

    per_part = [[ev[s][j][0].elapsed_time(ev[s][j][1]) / 1e3 for s in range(args.steps)] for j in range(len(parts))]
    step_s = sum(statistics.mean(x) for x in per_part)
    step_s_max = max_over_ranks(step_s, world)
    ideal = sum(p.ideal_s(peaks) for p in parts)
    value = job_value(ideal, step_s_max, world)

    detail = {}
    dom, dom_t = None, -1.0
    for p, ts in zip(parts, per_part):
        t = statistics.mean(ts)
        if p.kind == "paged_varlen":
            detail[p.name] = dict(ms=1e3 * t, ms_min=1e3 * min(ts), tflops=p.flops / t / 1e12, gbs=p.bytes / t / 1e9,
                                  frac=p.ideal_s(peaks) / t, gflop=p.flops / 1e9, gbytes=p.bytes / 1e9)
        elif p.kind in ("dense", "varlen"):
            ach = p.flops / t / 1e12
            detail[p.name] = dict(ms=1e3 * t, ms_min=1e3 * min(ts), tflops=ach,
                                  frac=ach / peaks["bf16_tflops"], gflop=p.flops / 1e9)
        else:
            ach = p.bytes / t / 1e9
            detail[p.name] = dict(ms=1e3 * t, ms_min=1e3 * min(ts), gbs=ach, frac=ach / peaks["hbm_gbs"],
                                  gbytes=p.bytes / 1e9)
        if t > dom_t:
            dom, dom_t = p, t
    if dom.kind == "paged_varlen":
        # one launch serving prefill chunks and decode steps: the roofline is
        # the sum of the FLOP term and the K/V byte term; the dominant one names it
        c = dom.data["config"]
        t_tensor = dom.flops / (peaks["bf16_tflops"] * 1e12)
        t_hbm = dom.bytes / (peaks["hbm_gbs"] * 1e9)
        if t_hbm >= t_tensor:
            roof = dict(bound="hbm", achieved=dom.bytes / dom_t / 1e9, peak=peaks["hbm_gbs"], unit="GB/s",
                        frac=dom.bytes / dom_t / 1e9 / peaks["hbm_gbs"])
        else:
            roof = dict(bound="tensor", achieved=dom.flops / dom_t / 1e12, peak=peaks["bf16_tflops"], unit="TFLOP/s",
                        frac=dom.flops / dom_t / 1e12 / peaks["bf16_tflops"])
        roof.update(kernel="onetile_kernel<%d,kPaged> + varlen_plan_kernel (%s)" % (c["D"], dom.name),
                    traffic=traffic_per_launch(dom), peak_source=peaks["source"],
                    mixed=dict(tflops=dom.flops / dom_t / 1e12, gbs=dom.bytes / dom_t / 1e9,
                               frac_of_summed_roofline=(t_tensor + t_hbm) / dom_t))
    elif dom.kind == "varlen":
        ach = dom.flops / dom_t / 1e12
        roof = dict(kernel="onetile_kernel<%d,kPacked> + varlen_plan_kernel (%s)" % (dom.data["config"]["D"], dom.name),
                    bound="tensor", achieved=ach, peak=peaks["bf16_tflops"], unit="TFLOP/s",
                    frac=ach / peaks["bf16_tflops"], traffic=traffic_per_launch(dom),
                    peak_source=peaks["source"] + " bf16 burst")
    elif dom.kind == "dense":
        ach = dom.flops / dom_t / 1e12
        kname = ("onetile_kernel<256,kBSHD>" if dom.data["config"]["D"] == 256
                 else "prefill_kernel<%d>" % dom.data["config"]["D"])
        roof = dict(kernel=kname + " (" + dom.name + ")", bound="tensor", achieved=ach,
                    peak=peaks["bf16_tflops"], unit="TFLOP/s", frac=ach / peaks["bf16_tflops"],
                    traffic=traffic_per_launch(dom), peak_source=peaks["source"] + " bf16 burst")
    else:
        ach = dom.bytes / dom_t / 1e9
        c = dom.data["config"]
        rows = c["Hq"] // c["Hkv"] * c["Sq"]
        tc = c["D"] in (128, 256) and 32 <= rows <= 128 and c["page_size"] % 8 == 0 and (
            c["page_size"] >= 64 or 64 % c["page_size"] == 0)
        mf = min(4, (rows + 15) // 16)
        split = "decode_tc_kernel<%d>" % c["D"] if tc else "decode_tma_kernel<%d,%d>" % (c["D"], mf)
        if dom.kind == "paged_fp8":
            split = ("decode_tc_kernel<%d,e4m3>" % c["D"]) if tc else "decode_fp8_kernel<%d,%d>" % (c["D"], mf)
        roof = dict(kernel=split + " + decode_combine_kernel<%d> (%s)" % (c["D"], dom.name), bound="hbm",
                    achieved=ach, peak=peaks["hbm_gbs"], unit="GB/s", frac=ach / peaks["hbm_gbs"],
                    traffic=traffic_per_launch(dom),
                    peak_source=peaks["source"] + " copy bandwidth")

    e2e = bench_e2e(args, parts, peaks, dev, stream, world)
    cpu = cpu_baseline(args, parts, peaks) if (rank == 0 and world == 1 and not args.no_cpu) else None

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * step_s_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        # the arithmetic type: e4m3fn caches widened to float16 products, else bf16
        "dtype": "e4m3kv-f16" if any(p.kind == "paged_fp8" for p in parts) else "bf16", "data": "synthetic",
        "config": {"workload": "serving step: qwen3_8b_prefill + paged_decode" if args.workload == "step"
                   else args.workload,
                   "parts": {p.name: p.data["config"] for p in parts}, "parallelism": "replicas",
                   "l2": "flushed between steps (%d MB write)" % (flush.numel() * 4 >> 20)},
        "parts": detail, "roofline": roof, "e2e": e2e, "cpu_baseline": cpu, "clocks": clk,
        "gpu_launches": args.steps * sum(p.launches() for p in parts),
        "peaks": peaks, "wall_s_timed_loop": wall,
    }
    return line


def bench_e2e(args, parts, peaks, dev, stream, world):
    """Same metric through the public calls with host-resident inputs: each step
    copies its inputs host->device (pinned) and its outputs back."""
    for p in parts:
        p.pin()
    steps = max(1, min(args.steps, args.e2e_steps))
    times, h2d, d2h = [], 0, 0
    for s in range(1 + steps):                  # one untimed warm-up
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d = sum(p.h2d() for p in parts)
        for p in parts:
            p.run()
        d2h = sum(p.d2h() for p in parts)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if s > 0:
            times.append(e0.elapsed_time(e1) / 1e3)
    t = max_over_ranks(statistics.mean(times), world)
    ideal = sum(p.ideal_s(peaks) for p in parts)
    return dict(value=job_value(ideal, t, world), unit=UNIT, ms_per_step=1e3 * t, h2d_bytes_per_step=h2d,
                d2h_bytes_per_step=d2h, steps=steps)


# --------------------------------------------------------------------------- oracle timing
def oracle_sample(parts, prefill_rows, decode_requests, seed=0):
    """Time the FP64 oracle on a bounded sample of each part; returns the
    estimated seconds for the whole step and a description of the sample."""
    import oracle
    est, desc = 0.0, []
    gen = torch.Generator().manual_seed(seed)
    for p in parts:
        d, c = p.data, p.data["config"]
        if p.kind == "dense":
            n = prefill_rows
            rows = torch.stack([torch.randint(0, c["B"], (n,), generator=gen),
                                torch.randint(0, c["Sq"], (n,), generator=gen),
                                torch.randint(0, c["Hq"], (n,), generator=gen)], 1)
            m = d["key_padding_mask"]
            pairs = 0
            for b, i, _h in rows.tolist():
                lim = max(0, min(c["Skv"], i + c["Skv"] - c["Sq"] + 1))
                pairs += int(m[b, :lim].sum()) if m is not None else lim
            t0 = time.perf_counter()
            oracle.attn_dense_rows(d["q"], d["k"], d["v"], rows.tolist(), key_padding_mask=m, causal=True)
            dt = time.perf_counter() - t0
            total_pairs = p.pairs * c["Hq"]            # p.pairs counts one head
            est += dt * total_pairs / max(pairs, 1)
            desc.append("%s: %d random rows (%.2f%% of its pairs) in %.2fs" % (p.name, n, 100.0 * pairs / total_pairs,
                                                                              dt))
        elif p.kind in ("varlen", "paged_varlen"):
            # random packed query rows, each as a one-query call whose keys end
            # at that query's position (end-aligned causal)
            n = max(1, prefill_rows // 64)
            cu = d["cu_seqlens_q"]
            tq = int(cu[-1])
            one = torch.tensor([0, 1], dtype=torch.int32)
            rows = torch.randint(0, tq, (n,), generator=gen).tolist()
            pairs, dt = 0, 0.0
            for t in rows:
                b = int(torch.searchsorted(cu, torch.tensor(t), right=True)) - 1
                sq, i = int(cu[b + 1] - cu[b]), t - int(cu[b])
                if p.kind == "varlen":
                    ks, L = int(d["cu_seqlens_kv"][b]), int(d["cu_seqlens_kv"][b + 1] - d["cu_seqlens_kv"][b])
                    vis = max(0, min(L, i + L - sq + 1))
                    t0 = time.perf_counter()
                    oracle.attn_varlen(d["q"][t:t + 1], d["k"][ks:ks + vis], d["v"][ks:ks + vis], one,
                                       torch.tensor([0, vis], dtype=torch.int32), causal=True)
                else:
                    L = int(d["cache_seqlens"][b])
                    vis = max(0, min(L, i + L - sq + 1))
                    t0 = time.perf_counter()
                    oracle.attn_paged_varlen(d["q"][t:t + 1], d["k_cache"], d["v_cache"], one,
                                             torch.tensor([vis], dtype=torch.int32), d["block_table"][b:b + 1],
                                             causal=True)
                dt += time.perf_counter() - t0
                pairs += vis
            est += dt * p.pairs / max(pairs, 1)
            desc.append("%s: %d random query rows (%.3f%% of its pairs) in %.2fs" % (p.name, n, 100.0 * pairs / p.pairs,
                                                                                    dt))
        else:
            n = min(decode_requests, c["B"])
            reqs = torch.randperm(c["B"], generator=gen)[:n].tolist()
            elem = 1 if p.kind == "paged_fp8" else 2
            sel_bytes = float(d["real_seqlen_kv"][reqs].to(torch.int64).sum()) * 2 * c["Hkv"] * c["D"] * elem
            t0 = time.perf_counter()
            if p.kind == "paged_fp8":
                oracle.attn_paged_fp8kv(d["q"], d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"],
                                        d["real_seqlen_kv"], d["block_table"], causal=True, requests=reqs)
            else:
                oracle.attn_paged(d["q"], d["k_cache"], d["v_cache"], d["real_seqlen_kv"], d["block_table"],
                                  causal=True, requests=reqs)
            dt = time.perf_counter() - t0
            est += dt * p.bytes / max(sel_bytes, 1.0)
            desc.append("%s: %d whole requests (%.2f%% of its bytes) in %.2fs" % (p.name, n, 100.0 * sel_bytes / p.bytes,
                                                                                  dt))
    return est, "; ".join(desc)


def oracle_whole(parts):
    """Time the FP64 oracle on the whole step (every row of every part)."""
    import oracle
    t0 = time.perf_counter()
    for p in parts:
        d = p.data
        if p.kind == "dense":
            oracle.attn_dense(d["q"], d["k"], d["v"], key_padding_mask=d["key_padding_mask"], causal=True)
        elif p.kind == "varlen":
            oracle.attn_varlen(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_kv"], causal=True)
        elif p.kind == "paged_varlen":
            oracle.attn_paged_varlen(d["q"], d["k_cache"], d["v_cache"], d["cu_seqlens_q"], d["cache_seqlens"],
                                     d["block_table"], causal=True)
        elif p.kind == "paged_fp8":
            oracle.attn_paged_fp8kv(d["q"], d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"],
                                    d["real_seqlen_kv"], d["block_table"], causal=True)
        else:
            oracle.attn_paged(d["q"], d["k_cache"], d["v_cache"], d["real_seqlen_kv"], d["block_table"], causal=True)
    return time.perf_counter() - t0


def cpu_baseline(args, parts, peaks):
    import oracle
    ideal = sum(p.ideal_s(peaks) for p in parts)
    if sum(p.flops for p in parts) < 2e12 and all(p.kind in ("dense", "paged", "paged_fp8") for p in parts):
        # the whole step takes seconds on the host cores
        est = oracle_whole(parts)
        desc = "the whole step (%s), every row, once" % " + ".join(p.name for p in parts)
    else:
        est, desc = oracle_sample(parts, args.cpu_rows, args.cpu_requests)
        desc = "sample scaled to the whole step: " + desc
    return dict(value=100.0 * ideal / est, unit=UNIT, cores=oracle.max_threads(), kind="oracle", sample=desc,
                step_s=est)


def bench_reference(args, world, rank):
    """The FP64 oracle as the reference arm: each step times a bounded sample of
    the workload on the host cores and scales it to the whole step."""
    if rank != 0:
        return None
    import oracle
    peaks = load_peaks()
    parts = make_parts(args.workload)
    for _ in range(args.warmup):
        oracle_sample(parts, 16, 1, seed=1000)
    ests = []
    descs = []
    for s in range(args.steps):
        est, desc = oracle_sample(parts, args.ref_rows, 1, seed=s)
        ests.append(est)
        descs.append(desc)
    est = statistics.mean(ests)
    ideal = sum(p.ideal_s(peaks) for p in parts)
    value = 100.0 * ideal / est
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * est, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "serving step: qwen3_8b_prefill + paged_decode" if args.workload == "step"
                   else args.workload, "parts": {p.name: p.data["config"] for p in parts}},
        "cpu_baseline": dict(kind="oracle", cores=oracle.max_threads(), value=value, unit=UNIT,
                             sample="per step: " + descs[0]),
        "e2e": dict(value=value, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0),
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="step", choices=["step"] + sorted(W.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-rows", type=int, default=4096)
    ap.add_argument("--cpu-requests", type=int, default=8)
    ap.add_argument("--ref-rows", type=int, default=64)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--batch", type=int, default=None, help="override B of a single named workload")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.batch is not None and args.workload == "step":
        ap.error("--batch applies to a single named workload")
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return
        else:
            dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.impl == "reference":
        line = bench_reference(args, world, rank)
    else:
        line = bench_ours(args, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line))
    if world > 1 and args.impl != "reference":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
