#!/usr/bin/env python
"""Benchmark of the causal GQA attention forward hot path on GB300.

One step = one pass of the whole path over the five synthetic workloads, each
through its own entry point (inputs resident in HBM before timing), in this
order:
  * long_chunked_prefill: B=4, Sq=2048 queries at the end of Skv=32768 keys,
    Hq=64, Hkv=8, D=128, causal, values N(0, 0.5^2);
  * qwen3_8b_prefill: dense prefill, B=2, Sq=Skv=4096, Hq=32, Hkv=8, D=128,
    causal, key_padding_mask with per-batch valid lengths U[2048, 4096];
  * tiny_dense: B=1, Hq=4, Hkv=2, Sq=Skv=128, D=64, causal (latency only);
  * paged_decode: B=64, Sq=1, Hq=32, Hkv=8, D=128, pages of 64 tokens, lengths
    U[1024, 16384], pages shuffled through block_table;
  * wide_group_decode: B=32, Sq=4 causal, Hq=24, Hkv=2, D=256, pages of 16
    tokens, lengths U[512, 32768].
Work is counted algorithmically: prefill FLOPs = 4 * D * Hq * (visible
query/key pairs), decode bytes = the K and V bytes of the real tokens (one byte
per element for e4m3fn caches).  The reported value is the step's roofline
efficiency, 100 * sum(FLOPs / tensor peak + bytes / HBM peak) / step time, with
the measured peaks of this machine; per-workload TFLOP/s or GB/s and their
fractions of the measured (and of the nominal) peaks are reported beside it.
Between timed steps a buffer twice the L2 size is overwritten so every step
starts with a cold L2.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload step|serving_step|<one workload name>]
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
# nominal GB300 figures: dense bf16 tensor peak and HBM3e bandwidth
NOMINAL = {"bf16_tflops": 2250.0, "hbm_gbs": 8000.0}
# The five-workload step runs the two prefill workloads first and back to back:
# they launch the same kernel instantiation, so the second finds its code in the
# SMs' instruction caches (a different large kernel in between, such as the
# D = 64 tiny call, costs the next launch about 10 us of instruction fetch).
STEPS = {
    "step": ["long_chunked_prefill", "qwen3_8b_prefill", "tiny_dense", "paged_decode", "wide_group_decode"],
    "serving_step": ["qwen3_8b_prefill", "paged_decode"],
}
# Roofline targets per workload, judged on the measured peaks: causal prefill
# at least 60 % of the dense bf16 tensor peak, paged decode at least 75 % of
# the HBM bandwidth.  tiny_dense is latency-bound and has none.
TARGETS = {"qwen3_8b_prefill": 0.60, "long_chunked_prefill": 0.60, "paged_decode": 0.75,
           "wide_group_decode": 0.75}


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


def executed_work(d, tile=128):
    """FLOPs the dense kernels execute: whole 128 x 128 (query, key) tiles, one
    query head at a time, for every tile holding at least one visible pair
    (the kernels skip the rest); the visible-pair count above is the work the
    roofline fractions use."""
    c = d["config"]
    B, Sq, Skv = c["B"], c["Sq"], c["Skv"]
    nq, nk = (Sq + tile - 1) // tile, (Skv + tile - 1) // tile
    m = d["key_padding_mask"]
    if m is None:
        any_key = torch.ones(B, nk, dtype=torch.bool)
    else:
        pad = torch.zeros(B, nk * tile, dtype=torch.bool)
        pad[:, :Skv] = m.to(torch.bool)
        any_key = pad.view(B, nk, tile).any(-1)
    kt = torch.arange(nk, dtype=torch.int64)
    tiles = 0
    for qt in range(nq):
        last = min(Skv - 1, (qt + 1) * tile - 1 + Skv - Sq) if c["causal"] else Skv - 1
        if last < 0:
            continue
        tiles += int((any_key & (kt * tile <= last)[None, :]).sum())
    return 4.0 * tile * tile * c["D"] * c["Hq"] * tiles


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
# reduced batch), for the prefill as bytes per launch of the same workload
# (long_chunked_prefill captured at B=1 of its four independent batches and
# scaled by 4).
TRAFFIC = {
    "tiny_dense": ("bytes", 236.54e3 + 0.0),
    "qwen3_8b_prefill": ("bytes", (94.029056 + 31.439360) * 1e6),
    "long_chunked_prefill": ("bytes", 4 * (534.310144 + 31.316480) * 1e6),
    "paged_decode": ("ratio", (559.379712 + 6.031616) / 556.916736),
    "wide_group_decode": ("ratio", (233.683200 + 3.794688) / 232.683520),
    "paged_decode_fp8kv": ("ratio", (279.798016 + 5.109504) / 278.458368),
    "wide_group_prefill": ("bytes", (235.305216 + 159.707392) * 1e6),
    "varlen_prefill": ("bytes", (799.823872 + 502.045696) * 1e6),
}


def traffic_per_launch(part):
    """DRAM bytes per launch from TRAFFIC; a fixed byte count holds only at the
    workload's own batch size."""
    t = TRAFFIC.get(part.name)
    if t is None:
        return None
    if t[0] == "ratio":
        return t[1] * part.bytes
    return t[1] if part.data["config"].get("B") == W.WORKLOADS[part.name].get("B") else None


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
            if self.kind == "varlen":
                need = g.attn_varlen_workspace_size(len(d["cu_seqlens_q"]) - 1, tq, c["Hq"], c["Hkv"])
            else:
                need = g.attn_paged_workspace_size(len(d["cu_seqlens_q"]) - 1, tq, c["Hq"], c["Hkv"], c["D"],
                                                   c["page_size"], d["block_table"].shape[1])
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

    def _routes_decode(self):
        """A mixed paged call whose one-query requests run on the split decode
        kernel (KV groups of fewer than 32 query heads)."""
        c = self.data["config"]
        return self.kind == "paged_varlen" and c["Hq"] // c["Hkv"] < 32

    def launches(self):
        # dense: one; packed: plan + attention (+ split decode + combine for a
        # mixed paged call); decode: split + combine
        if self.kind == "dense":
            return 1
        return 4 if self._routes_decode() else 2

    def bound(self, peaks):
        """"tensor" or "hbm": the larger of the FLOP and byte terms."""
        return "tensor" if self.flops / peaks["bf16_tflops"] / 1e12 >= self.bytes / peaks["hbm_gbs"] / 1e9 else "hbm"

    def kernel_name(self):
        """The kernels this part launches, as the profiler lists them."""
        c = self.data["config"]
        if self.kind == "dense":
            return "onetile_kernel<256,kBSHD>" if c["D"] == 256 else "prefill_kernel<%d>" % c["D"]
        if self.kind == "varlen":
            if c["D"] == 256:
                return "onetile_kernel<256,kPacked> + varlen_plan_kernel"
            return "prefill_kernel<%d,kModePacked> + varlen_plan_kernel" % c["D"]
        if self.kind == "paged_varlen":
            name = "onetile_kernel<%d,kPaged> + varlen_plan_kernel" % c["D"]
            if self._routes_decode():
                mf = min(4, (c["Hq"] // c["Hkv"] + 15) // 16)
                name = "decode_tma_kernel<%d,%d> + decode_combine_kernel<%d> + " % (c["D"], mf, c["D"]) + name
            return name
        rows = c["Hq"] // c["Hkv"] * c["Sq"]
        tc = c["D"] in (128, 256) and 32 <= rows <= 128 and c["page_size"] % 8 == 0 and (
            c["page_size"] >= 64 or 64 % c["page_size"] == 0)
        mf = min(4, (rows + 15) // 16)
        if self.kind == "paged_fp8":
            split = ("decode_tc_kernel<%d,e4m3>" % c["D"]) if tc else "decode_fp8_kernel<%d,%d>" % (c["D"], mf)
        else:
            split = "decode_tc_kernel<%d>" % c["D"] if tc else "decode_tma_kernel<%d,%d>" % (c["D"], mf)
        return split + " + decode_combine_kernel<%d>" % c["D"]

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
    names = STEPS.get(workload, [workload])
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


def workload_label(workload):
    if workload in STEPS:
        return "%s: %s" % ("five-workload step" if workload == "step" else "serving step",
                           " + ".join(STEPS[workload]))
    return workload


# --------------------------------------------------------------------------- clocks
class NvmlClocks:
    """SM clock, its maximum, power and the clock-event reasons, read through
    NVML (read-only queries) every few milliseconds on a host thread while the
    timed loop runs."""
    # nvml.h clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index, period_s=0.002):
        import ctypes
        import threading
        self.ct = ctypes
        self.period = period_s
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle for " + uuid)
        self.reason_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.sm_max = float(mx.value) if self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0 \
            else None
        self.rows = []
        self.stop_ev = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)

    def _sample(self):
        ct = self.ct
        clk, rs, pw = ct.c_uint(), ct.c_ulonglong(), ct.c_uint()
        ok = self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(clk)) == 0      # NVML_CLOCK_SM
        ok = ok and self.reason_fn(self.h, ct.byref(rs)) == 0
        p = pw.value / 1e3 if self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(pw)) == 0 else None
        if ok:
            self.rows.append((time.perf_counter(), float(clk.value), int(rs.value), p))

    def _run(self):
        while not self.stop_ev.is_set():
            self._sample()
            time.sleep(self.period)

    def start(self):
        self._sample()
        self.thread.start()

    def stop(self, t0, t1):
        self.stop_ev.set()
        self.thread.join()
        rows = [r for r in self.rows if t0 <= r[0] <= t1] or self.rows[-1:]
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for bit, name in self.REASONS.items():
                if r[2] & bit:
                    reasons.add(name)
        pw = [r[3] for r in rows if r[3] is not None]
        return dict(sm_mhz=statistics.median(r[1] for r in rows), sm_max_mhz=self.sm_max,
                    sm_mhz_min=min(r[1] for r in rows), reasons=sorted(reasons), samples=len(rows),
                    power_w_max=max(pw) if pw else None, source="NVML, every %g ms" % (1e3 * self.period))


class SmiClocks:
    """Fallback sampler: nvidia-smi every 50 ms."""
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

    def stop(self, t0=None, t1=None):
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
                    reasons=sorted(reasons), samples=len(rows), source="nvidia-smi, every 50 ms")


def clock_sampler(device_index):
    try:
        return NvmlClocks(device_index)
    except Exception:
        return SmiClocks(device_index)


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
def part_detail(p, ts, peaks):
    """Per-part timing: mean and min launch-group time, achieved rate and its
    fraction of the measured and of the nominal peak, the target if any."""
    t = statistics.mean(ts)
    d = dict(kernel=p.kernel_name(), ms=1e3 * t, ms_median=1e3 * statistics.median(ts), ms_min=1e3 * min(ts),
             bound=p.bound(peaks))
    if p.kind == "dense":
        ex = executed_work(p.data)
        d.update(executed_gflop=ex / 1e9, executed_tflops=ex / t / 1e12)
    if p.kind == "paged_varlen":
        d.update(tflops=p.flops / t / 1e12, gbs=p.bytes / t / 1e9, frac=p.ideal_s(peaks) / t,
                 gflop=p.flops / 1e9, gbytes=p.bytes / 1e9)
    elif p.flops > 0:
        ach = p.flops / t / 1e12
        d.update(tflops=ach, frac=ach / peaks["bf16_tflops"], frac_nominal=ach / NOMINAL["bf16_tflops"],
                 gflop=p.flops / 1e9)
    else:
        ach = p.bytes / t / 1e9
        d.update(gbs=ach, frac=ach / peaks["hbm_gbs"], frac_nominal=ach / NOMINAL["hbm_gbs"], gbytes=p.bytes / 1e9)
    if p.name in TARGETS:
        d.update(target=TARGETS[p.name], met=d["frac"] >= TARGETS[p.name])
    tr = traffic_per_launch(p)
    d["dram_traffic_bytes"] = tr
    return d


def roofline_of(p, t, peaks):
    """The roofline object of the dominant part (largest mean time)."""
    t_tensor = p.flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = p.bytes / (peaks["hbm_gbs"] * 1e9)
    if t_tensor >= t_hbm:
        ach = p.flops / t / 1e12
        roof = dict(bound="tensor", achieved=ach, peak=peaks["bf16_tflops"], unit="TFLOP/s",
                    frac=ach / peaks["bf16_tflops"], peak_source=peaks["source"] + " bf16 burst",
                    frac_of_sustained=ach / peaks["bf16_tflops_sustained"],
                    frac_nominal=ach / NOMINAL["bf16_tflops"])
    else:
        ach = p.bytes / t / 1e9
        roof = dict(bound="hbm", achieved=ach, peak=peaks["hbm_gbs"], unit="GB/s", frac=ach / peaks["hbm_gbs"],
                    peak_source=peaks["source"] + " copy bandwidth", frac_nominal=ach / NOMINAL["hbm_gbs"])
    roof.update(kernel="%s (%s)" % (p.kernel_name(), p.name), traffic=traffic_per_launch(p),
                algorithmic=dict(flops=p.flops, bytes=p.bytes))
    if p.kind == "paged_varlen":
        roof["mixed"] = dict(tflops=p.flops / t / 1e12, gbs=p.bytes / t / 1e9,
                             frac_of_summed_roofline=(t_tensor + t_hbm) / t)
    return roof


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
    clocks = clock_sampler(local)
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
    t1 = time.perf_counter()
    barrier(world)
    wall = time.perf_counter() - t0
    clk = clocks.stop(t0, t1)
    g.gqa_device_error()

    per_part = [[ev[s][j][0].elapsed_time(ev[s][j][1]) / 1e3 for s in range(args.steps)] for j in range(len(parts))]
    step_s = sum(statistics.mean(x) for x in per_part)
    step_s_max = max_over_ranks(step_s, world)
    ideal = sum(p.ideal_s(peaks) for p in parts)
    value = job_value(ideal, step_s_max, world)

    detail = {p.name: part_detail(p, ts, peaks) for p, ts in zip(parts, per_part)}
    dom_j = max(range(len(parts)), key=lambda j: statistics.mean(per_part[j]))
    roof = roofline_of(parts[dom_j], statistics.mean(per_part[dom_j]), peaks)

    graph = bench_graph(args, parts, flush, stream, dev)
    e2e = bench_e2e(args, parts, peaks, dev, stream, world)
    cpu = cpu_baseline(args, parts, peaks) if (rank == 0 and world == 1 and not args.no_cpu) else None

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * step_s_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        # the arithmetic type: e4m3fn caches widened to float16 products, else bf16
        "dtype": "e4m3kv-f16" if any(p.kind == "paged_fp8" for p in parts) else "bf16", "data": "synthetic",
        "config": {"workload": workload_label(args.workload),
                   "parts": {p.name: p.data["config"] for p in parts}, "parallelism": "replicas",
                   "l2": "flushed between steps (%d MB write)" % (flush.numel() * 4 >> 20)},
        "parts": detail, "roofline": roof, "graph_replay": graph, "e2e": e2e, "cpu_baseline": cpu, "clocks": clk,
        "targets": {"judged_on": "measured peaks (MEASURED_PEAKS.json); frac_nominal uses %g TFLOP/s and %g GB/s"
                                 % (NOMINAL["bf16_tflops"], NOMINAL["hbm_gbs"]),
                    "met": {n: d["met"] for n, d in detail.items() if "met" in d}},
        "gpu_launches": args.steps * sum(p.launches() for p in parts),
        "peaks": peaks, "wall_s_timed_loop": wall,
    }
    return line


def bench_graph(args, parts, flush, stream, dev):
    """The step's calls captured once in a CUDA graph and replayed `steps`
    times, L2 flushed before each replay (outside the events).  Outside the
    timed region of the headline value; a capture that fails is reported, not
    raised."""
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for p in parts:
                p.run()
        graph.replay()
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1))
        del graph
        return dict(ms_per_step=statistics.mean(ts), ms_median=statistics.median(ts), ms_min=min(ts),
                    replays=len(ts))
    except RuntimeError as e:
        return dict(error=str(e).splitlines()[0][:200])


def bench_e2e(args, parts, peaks, dev, stream, world):
    """Same metric through the public calls with host-resident inputs: each step
    copies its inputs host->device (pinned) and its outputs back.  The copies
    run on two side streams, inputs in the parts' order on one and outputs on
    the other (the link's two directions), so that a part's kernels start once
    its own inputs have landed and overlap the copies of the parts after it;
    the timed region spans every copy."""
    for p in parts:
        p.pin()
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    steps = max(1, min(args.steps, args.e2e_steps))
    times, h2d, d2h = [], 0, 0
    for s in range(1 + steps):                  # one untimed warm-up
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        up.wait_event(e0)
        down.wait_event(e0)
        landed = []
        h2d = d2h = 0
        with torch.cuda.stream(up):
            for p in parts:
                h2d += p.h2d()
                landed.append(torch.cuda.Event())
                landed[-1].record(up)
        for p, ev in zip(parts, landed):
            stream.wait_event(ev)
            p.run()
            done = torch.cuda.Event()
            done.record(stream)
            down.wait_event(done)
            with torch.cuda.stream(down):
                d2h += p.d2h()
        stream.wait_stream(up)
        stream.wait_stream(down)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if s > 0:
            times.append(e0.elapsed_time(e1) / 1e3)
    t = max_over_ranks(statistics.mean(times), world)
    ideal = sum(p.ideal_s(peaks) for p in parts)
    return dict(value=job_value(ideal, t, world), unit=UNIT, ms_per_step=1e3 * t, h2d_bytes_per_step=h2d,
                d2h_bytes_per_step=d2h, steps=steps)


# --------------------------------------------------------------------------- oracle timing
def _draw_sample(p, frac, gen):
    """A bounded random sample of part p: about `frac` of its work, at least
    one unit.  Units are query rows (b, i, h) of a dense call, query rows of
    a packed call, and (request, query head) pairs of a paged decode, whose K/V
    bytes count 1/g of that request's KV-head bytes (g query heads share them).
    Returns (kind of unit, units, sampled FLOPs, sampled bytes)."""
    d, c = p.data, p.data["config"]
    if p.kind == "dense":
        total = c["B"] * c["Sq"] * c["Hq"]
        n = max(1, min(total, int(round(frac * total))))
        flat = torch.randperm(total, generator=gen)[:n]
        rows = torch.stack([flat // (c["Sq"] * c["Hq"]), (flat // c["Hq"]) % c["Sq"], flat % c["Hq"]], 1).tolist()
        m = d["key_padding_mask"]
        pairs = 0
        for b, i, _h in rows:
            lim = max(0, min(c["Skv"], i + c["Skv"] - c["Sq"] + 1)) if c["causal"] else c["Skv"]
            pairs += int(m[b, :lim].sum()) if m is not None else lim
        return "rows", rows, 4.0 * c["D"] * pairs, 0.0
    if p.kind in ("varlen", "paged_varlen"):
        cu = d["cu_seqlens_q"]
        tq = int(cu[-1])
        n = max(1, int(round(frac * tq)))
        toks = torch.randperm(tq, generator=gen)[:n].tolist()
        units, flops, kvb = [], 0.0, 0.0
        for t in toks:
            b = int(torch.searchsorted(cu, torch.tensor(t), right=True)) - 1
            sq, i = int(cu[b + 1] - cu[b]), t - int(cu[b])
            L = (int(d["cu_seqlens_kv"][b + 1] - d["cu_seqlens_kv"][b]) if p.kind == "varlen"
                 else int(d["cache_seqlens"][b]))
            vis = max(0, min(L, i + L - sq + 1))
            units.append((t, b, vis))
            flops += 4.0 * c["D"] * c["Hq"] * vis
            if p.kind == "paged_varlen" and sq == 1:
                kvb += vis * 2 * c["Hkv"] * c["D"] * 2
        return "query rows", units, flops, kvb
    elem = 1 if p.kind == "paged_fp8" else 2
    g = c["Hq"] // c["Hkv"]
    lens = d["real_seqlen_kv"].tolist()
    want = frac * p.bytes
    units, got = [], 0.0
    for u in torch.randperm(c["B"] * c["Hq"], generator=gen).tolist():
        if units and got >= want:
            break
        b, h = divmod(u, c["Hq"])
        units.append((b, h))
        got += lens[b] * 2 * c["D"] * elem / g
    return "(request, query head) pairs", units, 0.0, got


def _decode_units(p, units):
    """The sampled (request, query head) pairs of a paged decode as one
    compact paged call with one query head and one KV head per request: each
    pair's pages (its KV head only) copied into a small pool in logical
    order.  Same arithmetic per row as the full call."""
    d, c = p.data, p.data["config"]
    ps, g = c["page_size"], c["Hq"] // c["Hkv"]
    lens = d["real_seqlen_kv"].tolist()
    kp, vp, tables, sl, qs, ks, vs = [], [], [], [], [], [], []
    first = 0
    for b, h in units:
        r = h // g
        n = max(1, -(-lens[b] // ps))
        pages = d["block_table"][b, :n].clamp(min=0).to(torch.int64)
        kp.append(d["k_cache"][pages][:, :, r:r + 1, :])
        vp.append(d["v_cache"][pages][:, :, r:r + 1, :])
        tables.append(list(range(first, first + n)))
        first += n
        sl.append(lens[b])
        qs.append(d["q"][b:b + 1, :, h:h + 1, :])
        if p.kind == "paged_fp8":
            ks.append(float(d["k_scale"][b, r]))
            vs.append(float(d["v_scale"][b, r]))
    width = max(len(t) for t in tables)
    bt = torch.full((len(units), width), -1, dtype=torch.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = torch.tensor(t, dtype=torch.int32)
    out = dict(q=torch.cat(qs).contiguous(), k_cache=torch.cat(kp).contiguous(), v_cache=torch.cat(vp).contiguous(),
               real_seqlen_kv=torch.tensor(sl, dtype=torch.int32), block_table=bt)
    if p.kind == "paged_fp8":
        out.update(k_scale=torch.tensor(ks).view(-1, 1), v_scale=torch.tensor(vs).view(-1, 1))
    return out


def _run_sample(p, unit, units, nthreads=0):
    """Run the FP64 oracle on a drawn sample; returns the seconds it took (the
    copy that gathers a decode sample's pages is not timed)."""
    import oracle
    d, c = p.data, p.data["config"]
    if p.kind in ("paged", "paged_fp8"):
        u = _decode_units(p, units)
        t0 = time.perf_counter()
        if p.kind == "paged_fp8":
            oracle.attn_paged_fp8kv(u["q"], u["k_cache"], u["v_cache"], u["k_scale"], u["v_scale"],
                                    u["real_seqlen_kv"], u["block_table"], causal=c["causal"], nthreads=nthreads)
        else:
            oracle.attn_paged(u["q"], u["k_cache"], u["v_cache"], u["real_seqlen_kv"], u["block_table"],
                              causal=c["causal"], nthreads=nthreads)
        return time.perf_counter() - t0
    t0 = time.perf_counter()
    if unit == "rows":
        oracle.attn_dense_rows(d["q"], d["k"], d["v"], units, key_padding_mask=d["key_padding_mask"],
                               causal=c["causal"], nthreads=nthreads)
    else:
        one = torch.tensor([0, 1], dtype=torch.int32)
        for t, b, vis in units:
            if p.kind == "varlen":
                ks = int(d["cu_seqlens_kv"][b])
                oracle.attn_varlen(d["q"][t:t + 1], d["k"][ks:ks + vis], d["v"][ks:ks + vis], one,
                                   torch.tensor([0, vis], dtype=torch.int32), causal=True, nthreads=nthreads)
            else:
                oracle.attn_paged_varlen(d["q"][t:t + 1], d["k_cache"], d["v_cache"], one,
                                         torch.tensor([vis], dtype=torch.int32), d["block_table"][b:b + 1],
                                         causal=True, nthreads=nthreads)
    return time.perf_counter() - t0


def oracle_sample(parts, peaks, frac, seed, nthreads=0):
    """Time the FP64 oracle on a bounded random sample of every part (about
    `frac` of each part's rows or K/V bytes).  Returns the sample's ideal
    seconds (its FLOPs and bytes at the measured peaks), the oracle's seconds
    on it, and per-part records."""
    gen = torch.Generator().manual_seed(seed)
    ideal, secs, recs = 0.0, 0.0, {}
    for p in parts:
        unit, units, flops, nbytes = _draw_sample(p, frac, gen)
        dt = _run_sample(p, unit, units, nthreads)
        i = flops / (peaks["bf16_tflops"] * 1e12) + nbytes / (peaks["hbm_gbs"] * 1e9)
        share = (flops / p.flops) if p.flops > 0 else (nbytes / p.bytes if p.bytes > 0 else 0.0)
        recs[p.name] = dict(sample="%d %s" % (len(units), unit), share_of_part=share, seconds=dt,
                            gflops_per_s=flops / dt / 1e9 if flops else None,
                            gbs=nbytes / dt / 1e9 if nbytes else None,
                            whole_part_s_est=dt / share if share > 0 else None)
        ideal += i
        secs += dt
    return ideal, secs, recs


def cpu_baseline(args, parts, peaks):
    """The FP64 oracle on the host cores, on a bounded sample of the step."""
    import oracle
    ideal, secs, recs = oracle_sample(parts, peaks, args.cpu_frac, seed=1)
    line = dict(value=100.0 * ideal / secs, unit=UNIT, cores=oracle.max_threads(), kind="oracle",
                sample="%.2f%% of each workload's rows or K/V bytes, drawn at random: %s" % (
                    100 * args.cpu_frac, "; ".join("%s %s" % (n, r["sample"]) for n, r in recs.items())),
                seconds=secs, step_s_est=secs * sum(p.ideal_s(peaks) for p in parts) / ideal, parts=recs)
    # one core against all cores on the same small sample of one prefill
    pf = [p for p in parts if p.kind == "dense" and p.flops > 1e9]
    if pf:
        p = pf[0]
        unit, units, flops, _ = _draw_sample(p, args.cpu_frac / 8, torch.Generator().manual_seed(2))
        t_all = _run_sample(p, unit, units, 0)
        t_one = _run_sample(p, unit, units, 1)
        line["one_core"] = dict(part=p.name, sample="%d %s" % (len(units), unit), gflop=flops / 1e9,
                                seconds_1_core=t_one, seconds_all_cores=t_all,
                                gflops_per_s_1_core=flops / t_one / 1e9, speedup=t_one / t_all)
    return line


def bench_reference(args, world, rank):
    """The FP64 oracle as the reference arm: each step times the oracle on a
    bounded random sample of the step's work (a fresh draw per step); the
    value is the sample's ideal time over the oracle's measured time, and
    ms_per_step is that measured time."""
    if rank != 0:
        return None
    import oracle
    peaks = load_peaks()
    parts = make_parts(args.workload)
    for w in range(args.warmup):
        oracle_sample(parts, peaks, args.ref_frac / 8, seed=1000 + w)
    ideals, secs, descs = [], [], None
    for s in range(args.steps):
        i, t, recs = oracle_sample(parts, peaks, args.ref_frac, seed=s)
        ideals.append(i)
        secs.append(t)
        descs = descs or recs
    value = 100.0 * sum(ideals) / sum(secs)
    ms = 1e3 * statistics.mean(secs)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_label(args.workload), "parts": {p.name: p.data["config"] for p in parts}},
        "cpu_baseline": dict(kind="oracle", cores=oracle.max_threads(), value=value, unit=UNIT,
                             sample="per step, a fresh random draw of %.2f%% of each workload's rows or K/V "
                                    "bytes (first step: %s)" % (100 * args.ref_frac, "; ".join(
                                        "%s %s" % (n, r["sample"]) for n, r in descs.items()))),
        "e2e": dict(value=value, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0),
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="step", choices=sorted(STEPS) + sorted(W.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-frac", type=float, default=0.02,
                    help="share of each workload the cpu_baseline times on the oracle")
    ap.add_argument("--ref-frac", type=float, default=0.004,
                    help="share of each workload one reference-arm step times on the oracle")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--batch", type=int, default=None, help="override B of a single named workload")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.batch is not None and args.workload in STEPS:
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
