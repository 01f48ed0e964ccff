#!/usr/bin/env python
"""bench.py — throughput of the paged-KV attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl pka|reference]

Prints ONE JSON line (rank 0).  A step is one pass of the hot path over one
batch of seeded synthetic input, already resident in HBM:

  t5-small-decode (default)  each sequence's new token appended to the cache
        and the biased paged decode, in one launch: 64 seqs x 8 heads x 64,
        bf16, contexts U[1,512], T5 bias [64,8,512] materialised from an
        [8,129] table.
  tiny-decode        4 x 2 x 64 fp32, contexts U[1,64], Gaussian bias.
  t5-large-decode    decoder self-attention (256 x 16 x 64 bf16, contexts
        U[1,2048], T5 bias padded to 2048) + encoder cross-attention (own block
        table, encoder length 512, no bias), in one launch that also appends
        the decoder's new token (the encoder cache is static).
  --separate-launches: reshape_and_cache of every side's new token, then one
        decode launch per side (the unfused step).
  long-ctx-decode    512 x 16 x 128 fp16, contexts log-U[16,8192], causal
        window 4096, bias [512,16,8192] N(0,0.25) NaN-padded.
  encoder-prefill    32 packed sequences U[128,8192], 12 heads x 64 bf16,
        three layers: full, window 64, window 64 (bidirectional); with
        --head-dim 128 the same shapes at head dim 128.
  chunked-prefill    the same sequences, one chunked-local layer (chunks of
        1024 positions, causal within the chunk).
  t5-encoder-prefill T5-large-shaped encoder self-attention: 256 x 512 tokens,
        16 heads x 64 bf16, bidirectional, T5 relative-position bias from a
        [16, 257] table computed in the kernel.
  t5-paged-prefill   a prompt chunk (the last min(ctx, U[1,256]) positions) of
        every sequence of the t5-large-decode batch through the block tables:
        its K/V written by reshape_and_cache, then causal + T5 bias over the
        self-attention cache, and unmasked over the encoder cache.

metric/unit: decode workloads report algorithmic KV+bias bytes per second
(GB/s); the prefill workload reports TFLOP/s (4*D per kept (query, key) pair
per head).  Inputs smaller than 3x L2 are rotated over enough copies that
every step reads cold data.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload, in the same unit.
N > 1 (torchrun): every rank runs its own replica (weak scaling; no
collective on the data path); time = max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth import BF16, F16, F32, ELT_BYTES  # noqa: E402

METRIC = "decode KV+bias GB/s (% of HBM peak) and seqs/sec, bias on/off; prefill TFLOPS"
L2_BYTES = 129 * 1024 * 1024
DECODE_WORKLOADS = {"tiny-decode": 1, "t5-small-decode": 2, "t5-large-decode": 3, "long-ctx-decode": 5}


# ---------------------------------------------------------------------------
# plumbing
# ---------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


def kernel_source_hash(name: str) -> str:
    """sha1[:12] of a kernel source with its comments, blank lines and each
    line's leading and trailing blanks removed (a comment edit leaves the
    recorded counters valid; a code edit does not)."""
    path = os.path.join(ROOT, "paged_kv_attention_23_gb300", "csrc", name)
    src = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
    lines = [re.sub(r"//.*$", "", ln).strip() for ln in src.splitlines()]
    code = "\n".join(ln for ln in lines if ln)
    return hashlib.sha1(code.encode()).hexdigest()[:12]


def recorded_traffic(kernel_file: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None if the
    kernel source changed since it was captured."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    h = kernel_source_hash(kernel_file)
    for line in open(p):
        f = line.split()
        if len(f) >= 4 and not line.startswith("#") and f[0] == kernel_file and f[1] == workload and f[3] == h:
            return float(f[2])
    return None


def gpu_id(local: int) -> str:
    """nvidia-smi's id of this rank's GPU (index or UUID)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x.strip() for x in vis.split(",") if x.strip()]
    return ids[local] if local < len(ids) else str(local)


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled every 200 ms."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0])); mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# decode workloads
# ---------------------------------------------------------------------------
def decode_alg_bytes(case, bias_on: bool, t5_table: bool = False) -> dict:
    """Algorithmic bytes of one decode call: visible K and V rows, bias
    entries of visible keys (or, with the T5 table computed in the kernel,
    the table), q and out rows, block-table entries, context lengths."""
    n = case.visible().astype(np.int64)
    H, D, elt = case.num_heads, case.head_dim, ELT_BYTES[case.dtype]
    kv = int((2 * H * n * D * elt).sum())
    if bias_on and t5_table and case.bias_table is not None:
        bias = int(case.bias_table.size * 4)
    else:
        bias = int((4 * H * n).sum()) if (bias_on and case.bias is not None) else 0
    other = int(case.num_seqs * 2 * H * D * elt + (4 * ((n + case.block_size - 1) // case.block_size)).sum()
                + 4 * case.num_seqs)
    return {"kv": kv, "bias": bias, "other": other, "total": kv + bias + other}


def _tdt(code):
    import torch
    return {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}[code]


def _dev(arr, code, device):
    import torch
    a = np.ascontiguousarray(arr)
    if code == BF16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def capture_graph(fn):
    """Capture fn()'s launches (all on the current stream) into a CUDA graph."""
    import torch
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    return g


def queue_ahead():
    """A GPU-side sleep (~0.5 ms) ahead of a timed region: the host submits the
    timed graph while it runs, so the region's events bracket device work only,
    not the host's graph-launch latency."""
    import torch
    torch.cuda._sleep(int(1e6))


def per_launch_ms(run, nsides, K):
    """Mean device duration of each side's timed launch over K steps: run(ev)
    records ev[side][0][k] / ev[side][1][k] around the launch of step k."""
    import torch
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(K)] for _ in range(2)] for _ in range(nsides)]
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e6) * (K + 10))          # ~1 ms per step at 2 GHz: the host queues ahead
    run(ev)
    torch.cuda.synchronize()
    return [statistics.mean(ev[j][0][k].elapsed_time(ev[j][1][k]) for k in range(K)) for j in range(nsides)]


class DecodeSide:
    """One decode call's device state (one attention type), with its new-token
    inputs for reshape_and_cache."""

    def __init__(self, case, pka, device):
        import torch
        self.case = case
        H, D, bs = case.num_heads, case.head_dim, case.block_size
        tdt = _tdt(case.dtype)
        if case.device_kv is not None:
            key, value = case.device_kv
        else:
            key, value = _dev(case.key, case.dtype, device), _dev(case.value, case.dtype, device)
        self.kc = torch.zeros((case.num_blocks, H, bs, D), dtype=tdt, device=device)
        self.vc = torch.zeros_like(self.kc)
        pka.reshape_and_cache(key, value, self.kc, self.vc, torch.from_numpy(case.slot_mapping).to(device))
        # the step's new token per sequence = its last context position
        last = np.where(case.context_lens > 0, case.tok_offsets[1:] - 1, 0)
        idx = torch.from_numpy(last.astype(np.int64)).to(device)
        self.new_k = key[idx].contiguous()
        self.new_v = value[idx].contiguous()
        slots = (np.where(case.context_lens > 0, case.slot_mapping[last], -1) if case.num_tokens
                 else np.full(case.num_seqs, -1))
        self.slots = torch.from_numpy(slots.astype(np.int64)).to(device)
        self.q = _dev(case.q, case.dtype, device)
        self.bt = torch.from_numpy(np.ascontiguousarray(case.block_tables)).to(device)
        self.cl = torch.from_numpy(case.context_lens).to(device)
        self.bias = torch.from_numpy(case.bias).to(device) if case.bias is not None else None
        self.table = (torch.from_numpy(case.bias_table).to(device) if getattr(case, "bias_table", None) is not None
                      else None)
        self.use_table = False
        self.append = True            # the step appends the newest token (not for the static encoder cache)
        self.out = torch.empty((case.num_seqs, H, D), dtype=tdt, device=device)
        self.ws = torch.zeros(pka.paged_attn_decode_workspace_size(case.num_seqs, H, D, case.max_context_len,
                                                                   case.window), dtype=torch.uint8, device=device)
        del key, value

    def clone(self):
        import copy
        c = copy.copy(self)
        for n in ("kc", "vc", "new_k", "new_v", "slots", "q", "bt", "cl", "out"):
            setattr(c, n, getattr(self, n).clone())
        c.bias = self.bias.clone() if self.bias is not None else None
        c.table = self.table.clone() if self.table is not None else None
        return c

    def nbytes(self):
        ts = [self.kc, self.vc, self.q, self.bt, self.new_k, self.new_v] + ([self.bias] if self.bias is not None else [])
        return sum(t.numel() * t.element_size() for t in ts)

    def reshape(self, pka):
        pka.reshape_and_cache(self.new_k, self.new_v, self.kc, self.vc, self.slots)

    def problem(self, bias_on=True):
        """This side as one problem of the fused launch."""
        c = self.case
        pr = dict(out=self.out, q=self.q, k_cache=self.kc, v_cache=self.vc, block_tables=self.bt, context_lens=self.cl,
                  sliding_window=c.window, scale=c.scale, max_context_len=c.max_context_len, workspace=self.ws)
        if self.append:
            pr["key_new"], pr["value_new"] = self.new_k, self.new_v
        if bias_on and self.use_table and self.table is not None:
            pr["bias_table"] = self.table
        elif bias_on and self.bias is not None:
            pr["attn_bias"] = self.bias
        return pr

    def decode(self, pka, bias_on=True):
        c = self.case
        if bias_on and self.use_table and self.table is not None:
            pka.paged_attn_decode_t5bias(self.out, self.q, self.kc, self.vc, self.bt, self.cl, self.table, c.window,
                                         c.scale, max_context_len=c.max_context_len, workspace=self.ws)
            return
        pka.paged_attn_decode(self.out, self.q, self.kc, self.vc, self.bt, self.cl,
                              self.bias if bias_on else None, c.window, c.scale, max_context_len=c.max_context_len,
                              workspace=self.ws)


def decode_all(pka, sides, fused, bias_on=True, events=None, k=0):
    """The step: fused, one launch that appends each appending side's newest
    token and decodes all sides; else reshape_and_cache of every side's new
    token, then one decode launch per side.  events[j] brackets decode launch j."""
    if not fused:
        for s in sides:
            s.reshape(pka)
    if fused:
        if events is not None:
            events[0][0][k].record()
        pka.paged_attn_decode_multi([s.problem(bias_on and s.bias is not None) for s in sides])
        if events is not None:
            events[0][1][k].record()
        return
    for j, s in enumerate(sides):
        if events is not None:
            events[j][0][k].record()
        s.decode(pka, bias_on and s.bias is not None)
        if events is not None:
            events[j][1][k].record()


def rot_sides_cross(rot):
    """The cross-attention side of every rotated copy (the second side)."""
    return [sides[1] for sides in rot]


def build_decode_sides(workload, device, on_device_draw, num_seqs=None):
    n = DECODE_WORKLOADS[workload]
    dev = device if on_device_draw else None
    cases = [synth.decode_workload(n, device=dev, num_seqs=num_seqs)]
    if n == 3:
        cases.append(synth.cross_workload(device=dev, num_seqs=num_seqs))
    return cases


def graph_ms(fn, K, world=1):
    """Mean device time of one fn(k), k < K: the K calls are captured into one
    CUDA graph, uploaded by an untimed replay, and one replay is timed with CUDA
    events queued behind a GPU-side sleep (the region holds device work only)."""
    import torch
    g = capture_graph(lambda: [fn(k) for k in range(K)])
    g.replay()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(); barrier(world)
    queue_ahead()
    t0.record()
    g.replay()
    t1.record()
    torch.cuda.synchronize(); barrier(world)
    ms = max_over_ranks(t0.elapsed_time(t1), world) / K
    del g
    return ms


class DecodeBench:
    """A decode workload resident on the device: its sides (self-attention,
    and cross-attention for the T5-large step), rotated over enough input
    copies that every step reads cold data."""

    def __init__(self, workload, pka, device, num_seqs=None, t5_table=False, keep_tokens=False):
        import torch
        self.workload = workload
        self.pka = pka
        big = workload in ("t5-large-decode", "long-ctx-decode")
        self.cases = build_decode_sides(workload, device, big, num_seqs)
        self.sides = [DecodeSide(c, pka, device) for c in self.cases]
        for sd in self.sides:
            sd.use_table = t5_table
        if not keep_tokens:
            for c in self.cases:          # the token arrays are only needed again by the CPU leg
                c.device_kv = None
            torch.cuda.empty_cache()
        self.t5_table = t5_table
        self.bytes_on = [decode_alg_bytes(c, True, t5_table) for c in self.cases]
        self.bytes_off = [decode_alg_bytes(c, False) for c in self.cases]
        self.per_copy = sum(s.nbytes() for s in self.sides)
        self.copies = max(1, min(16, math.ceil(3 * L2_BYTES / self.per_copy)))
        self.rot = [self.sides] + [[s.clone() for s in self.sides] for _ in range(self.copies - 1)]
        if len(self.sides) > 1:
            for s in rot_sides_cross(self.rot):
                s.append = False
        torch.cuda.synchronize()

    @property
    def has_bias(self):
        return any(s.bias is not None for s in self.sides)

    def step(self, k, bias_on=True, fused=True, events=None):
        decode_all(self.pka, self.rot[k % self.copies], fused, bias_on, events, k)

    def total(self, bias_on):
        return sum(b["total"] for b in (self.bytes_on if bias_on else self.bytes_off))

    def l2_note(self):
        return (f"inputs rotated over {self.copies} copies ({self.per_copy * self.copies / 2**20:.0f} MiB > L2)"
                if self.copies > 1 else f"inputs {self.per_copy / 2**20:.0f} MiB > L2")

    def record(self, K, peaks, world=1):
        """Graph-timed launch times of the step, bias on and off, each side's
        own launch for a two-sided step, and the bytes / fractions they give."""
        seqs = self.cases[0].num_seqs
        hbm = peaks["hbm_gbs"]

        def entry(ms, nbytes, nseqs):
            return {"ms_per_launch": round(ms, 5), "GBps": round(nbytes / (ms * 1e-3) / 1e9, 1),
                    "frac": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 4), "seqs_per_s": round(nseqs / (ms * 1e-3), 1),
                    "alg_bytes": nbytes}

        rec = {"launch": ("one launch: newest token appended + decode" +
                          (" of self and cross" if len(self.sides) > 1 else ""))}
        for on in ((True, False) if self.has_bias else (True,)):
            ms = graph_ms(lambda k: self.step(k, on), K, world)
            rec["bias_on" if on else "bias_off"] = entry(ms, self.total(on), seqs)
        if not self.has_bias:
            rec["bias_off"] = rec["bias_on"]
        if len(self.sides) > 1:
            names = ["self", "cross"]
            for j, sd in enumerate(self.sides):
                for on in ((True, False) if sd.bias is not None else (True,)):
                    ms = graph_ms(lambda k: self.rot[k % self.copies][j].decode(self.pka, on), K, world)
                    b = (self.bytes_on if on else self.bytes_off)[j]["total"]
                    key = f"{names[j]}_separate_launch" + ("" if sd.bias is None else
                                                             ("_bias_on" if on else "_bias_off"))
                    rec[key] = entry(ms, b, self.cases[j].num_seqs)
        return rec


def run_decode(args, rank, world, local, peaks):
    import torch
    import paged_kv_attention_23_gb300 as pka
    pka.load()
    device = f"cuda:{local}"
    torch.cuda.set_device(local)
    db = DecodeBench(args.workload, pka, device, args.num_seqs, args.t5_table)
    cases, sides = db.cases, db.sides
    fused = not args.separate_launches
    nlaunch = 1 if fused else len(sides)
    step_bytes = db.total(True)

    def step(i, bias_on=True, events=None):
        db.step(i, bias_on, fused, events)

    clocks = ClockSampler(gpu_id(local))
    clocks.start()
    t_end = time.time() + args.clock_soak                       # clock soak (untimed)
    i = 0
    while time.time() < t_end:
        step(i); i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    for w in range(args.warmup):
        step(w)
    K = args.steps
    # the K timed steps are one CUDA graph (no host launch gaps); one untimed
    # replay first uploads it
    graph = capture_graph(lambda: [step(k) for k in range(K)])
    graph.replay()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(); barrier(world)
    queue_ahead()
    t0.record()
    graph.replay()
    t1.record()
    torch.cuda.synchronize(); barrier(world)
    total_ms = max_over_ranks(t0.elapsed_time(t1), world)
    ms_step = total_ms / K
    del graph
    # bias off, timed the same way (one graph of K steps)
    off_ms = graph_ms(lambda k: step(k, False), K, world) if db.has_bias else None
    clk = clocks.stop()
    # warm-L2 reference (labelled, not the metric): the same steps on one input copy
    warm_ms = graph_ms(lambda k: step(0), K, world) if db.copies > 1 else None
    # per-launch durations by event pairs (labelled; they add a few microseconds
    # of their own to a short launch), and, for separate launches, each side's
    # launch graph-timed on its own
    launch_ms = per_launch_ms(lambda ev: [step(k, True, ev) for k in range(K)], nlaunch, K)
    bytes_on, bytes_off = db.bytes_on, db.bytes_off
    if fused:                          # one launch carries every side's bytes
        bytes_on = [{k: sum(b[k] for b in bytes_on) for k in bytes_on[0]}]
        bytes_off = [{k: sum(b[k] for b in bytes_off) for k in bytes_off[0]}]
        graph_launch_ms = [ms_step]
    else:
        graph_launch_ms = [graph_ms(lambda k: db.rot[k % db.copies][j].decode(pka, True), K, world)
                           for j in range(len(sides))]

    value = step_bytes * world / (ms_step * 1e-3) / 1e9
    # dominant kernel: the decode launch carrying the most bytes, its average
    # duration from a graph of its launches alone (the fused step is one launch)
    jd = int(np.argmax([b["total"] for b in bytes_on]))
    launch_avg_ms = graph_launch_ms[jd]
    achieved = bytes_on[jd]["total"] / (launch_avg_ms * 1e-3) / 1e9
    traffic = recorded_traffic("paged_decode.cu", args.workload)
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
            "kernel": "paged_decode_kernel", "alg_bytes_per_launch": bytes_on[jd]["total"],
            "launch_ms": round(launch_avg_ms, 5),
            "launch_timing": ("timed graph region / steps (one launch per step)" if fused
                              else "a graph of that launch alone / launches"),
            "launch_ms_event_pairs": round(launch_ms[jd], 5), "peak_src": peaks["src"] + " hbm_gbs (copy)"}
    e2e = decode_e2e(args, sides, pka, step_bytes, world, fused) if not args.no_e2e else None
    seqs = cases[0].num_seqs
    off_bytes = db.total(False)
    extra = {
        "bias_on": {"ms_per_step": round(ms_step, 5), "GBps": round(value / world, 1),
                    "frac": round(step_bytes / (ms_step * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                    "kv_GBps": round(sum(b["kv"] for b in db.bytes_on) / (ms_step * 1e-3) / 1e9, 1),
                    "seqs_per_s": round(seqs / (ms_step * 1e-3), 1), "alg_bytes": step_bytes},
        "bias_off": ({"ms_per_step": round(off_ms, 5), "GBps": round(off_bytes / (off_ms * 1e-3) / 1e9, 1),
                      "frac": round(off_bytes / (off_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                      "seqs_per_s": round(seqs / (off_ms * 1e-3), 1), "alg_bytes": off_bytes}
                     if off_ms else None),
        "timing": "bias on and off: one CUDA graph of the K steps each, cold L2",
        "decode_ms_per_launch_graph": [round(x, 5) for x in graph_launch_ms],
        "decode_ms_per_launch_event_pairs": [round(x, 5) for x in launch_ms],
        "warm_l2_GBps": round(step_bytes * world / (warm_ms * 1e-3) / 1e9, 1) if warm_ms else None,
        "warm_l2_ms_per_step": round(warm_ms, 5) if warm_ms else None,
    }
    cfg = {"workload": args.workload, "num_seqs": [c.num_seqs for c in cases], "num_heads": cases[0].num_heads,
           "head_dim": cases[0].head_dim, "block_size": 16,
           "window": [c.window for c in cases],
           "bias": [("t5 table in kernel" if args.t5_table and c.bias_table is not None else "materialised")
                    if c.bias is not None else None for c in cases],
           "l2": db.l2_note(), "parallelism": f"replicas x{world}",
           "launches_per_step": ("one: append of the newest token + decode" + (" of self and cross" if len(sides) > 1 else ""))
           if fused else "reshape_and_cache per side, then one decode per side"}
    res = {"value": value, "unit": "GB/s", "ms_per_step": ms_step, "dtype": synth.DTYPE_NAMES[cases[0].dtype],
           "config": cfg, "roofline": roof, "e2e": e2e, "clocks": clk,
           "gpu_launches": K * (1 if fused else 2 * len(sides)), "extra": extra}
    if not args.separate_launches and not args.t5_table and args.num_seqs is None:
        res["record"] = db.record(K, peaks, world) if args.per_config else None
    del db, sides, cases
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


PIPELINE_BYTES = 8 << 20    # decode e2e: steps that copy at least this much overlap copies and calls


def decode_e2e(args, sides, pka, step_bytes, world, fused=False):
    """The same step through the public API from pinned host buffers: copy the
    step's inputs host->device, run it, read the output back.  The inputs sit
    in one pinned staging buffer whose device twin holds every input tensor of
    the step (as a serving engine stages a step), so a step is one
    host->device copy, the call, and one device->host copy of the outputs.
    When a step copies at least PIPELINE_BYTES, steps alternate between two
    device twins: step k+1's inputs are copied on a second stream while step k
    computes, once step k-1 (the last reader of that twin) has finished.  A
    smaller step is bound by host calls, not by the copy, and runs copy, call,
    copy on one stream.  Every step copies all of its inputs and reads back its
    output inside the timed region."""
    import torch
    dev = sides[0].out.device
    fields = []
    for s in sides:
        names = (["q", "new_k", "new_v", "bt", "cl"] if s.append else ["q", "bt", "cl"]) if fused else \
            ["q", "new_k", "new_v", "slots", "bt", "cl"]
        if s.use_table and s.table is not None:
            names.append("table")
        elif s.bias is not None:
            names.append("bias")
        fields += [(s, n) for n in names]

    def stage(tensors):
        offs, total = [], 0
        for t in tensors:
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, total

    def view(buf, off, t):
        n = t.numel() * t.element_size()
        return buf[off:off + n].view(t.dtype).view(t.shape)

    saved = [(s, n, getattr(s, n)) for s, n in fields] + [(s, "out", s.out) for s in sides]
    offs, h2d = stage([getattr(s, n) for s, n in fields])
    h_in = torch.empty(h2d, dtype=torch.uint8, pin_memory=True)
    d_in = [torch.empty(h2d, dtype=torch.uint8, device=dev) for _ in range(2)]
    for (s, n), off in zip(fields, offs):
        view(h_in, off, getattr(s, n)).copy_(getattr(s, n))
    in_views = [[view(d, off, getattr(s, n)) for (s, n), off in zip(fields, offs)] for d in d_in]
    ooffs, d2h = stage([s.out for s in sides])
    h_out = torch.empty(d2h, dtype=torch.uint8, pin_memory=True)
    d_out = torch.empty(d2h, dtype=torch.uint8, device=dev)
    for s, off in zip(sides, ooffs):
        s.out = view(d_out, off, s.out)
    comp = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    pipelined = h2d >= PIPELINE_BYTES
    if not pipelined:
        for (s, n), v in zip(fields, in_views[0]):
            setattr(s, n, v)

    def step(k):
        if not pipelined:
            d_in[0].copy_(h_in, non_blocking=True)
            decode_all(pka, sides, fused)
            h_out.copy_(d_out, non_blocking=True)
            return
        j = k & 1
        with torch.cuda.stream(copy):
            if k >= 2:
                copy.wait_event(done[j])          # step k-2 has read this twin
            d_in[j].copy_(h_in, non_blocking=True)
            copied[j].record(copy)
        comp.wait_event(copied[j])
        for (s, n), v in zip(fields, in_views[j]):
            setattr(s, n, v)
        decode_all(pka, sides, fused)
        done[j].record(comp)
        h_out.copy_(d_out, non_blocking=True)

    try:
        for k in range(args.warmup):
            step(k)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(); barrier(world)
        a.record(comp)
        copy.wait_event(a)                        # the first copy starts inside the timed region
        for k in range(args.steps):
            step(k)
        b.record(comp)
        torch.cuda.synchronize(); barrier(world)
    finally:
        for s, n, t in saved:
            setattr(s, n, t)
    ms = max_over_ranks(a.elapsed_time(b), world) / args.steps
    return {"value": round(step_bytes * world / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 5),
            "copies": ("step k+1's inputs copied on a second stream while step k computes (two device twins)"
                       if pipelined else "copy, call, copy on one stream")}


# ---------------------------------------------------------------------------
# prefill workload
# ---------------------------------------------------------------------------
def prefill_flops(case) -> int:
    return 4 * case.head_dim * case.num_heads * case.visible_pairs()


PREFILL_WORKLOADS = ("encoder-prefill", "chunked-prefill", "t5-encoder-prefill", "t5-paged-prefill")


class PrefillLaunch:
    """One prefill call of a step: its device inputs, output and FLOPs.
    ``host_inputs`` are the tensors a step copies from the host for e2e."""

    def __init__(self, name, case, fn, out, flops, host_inputs, pre=None, nbytes=None):
        self.name, self.case, self.fn, self.out, self.flops = name, case, fn, out, flops
        self.nbytes = nbytes    # algorithmic HBM bytes of one launch
        self.host_inputs = host_inputs
        self.pre = pre               # work the step does before the call (reshape_and_cache of new K/V)

    def __call__(self):
        if self.pre is not None:
            self.pre()
        self.fn()


def packed_prefill_bytes(c) -> int:
    """Algorithmic bytes of a packed prefill layer: q, k, v read once, out
    written once (2-byte elements), and the bias table if any."""
    nbytes = 4 * c.num_tokens * c.num_heads * c.head_dim * 2
    if c.rel_bias is not None:
        nbytes += c.rel_bias.size * 4
    return nbytes


def paged_prefill_bytes(pc) -> int:
    """Algorithmic bytes of a paged prefill call: q read and out written once,
    and for every sequence and head the K and V rows its queries can see (the
    last query sees keys up to ctx - 1; a window starts the first query's keys
    W - 1 before it), the block-table entries of those rows, the context
    lengths and query offsets, and the bias table if any."""
    c = pc.cache
    H, D = pc.num_heads, pc.head_dim
    ctx = c.context_lens.astype(np.int64)
    lq = pc.query_lens.astype(np.int64)
    lo = np.zeros_like(ctx) if pc.window <= 0 else np.maximum(0, ctx - lq - pc.window + 1)
    keys = np.where(lq > 0, ctx - lo, 0)
    blocks = np.where(keys > 0, (ctx + 15) // 16 - lo // 16, 0)
    nbytes = int(keys.sum()) * H * D * 2 * 2 + 2 * int(lq.sum()) * H * D * 2
    nbytes += int(blocks.sum()) * 4 + 4 * len(ctx) + 4 * (len(ctx) + 1)
    if pc.rel_bias is not None:
        nbytes += pc.rel_bias.size * 4
    return nbytes


def prefill_bound(flops, nbytes, ms, peaks):
    """The roofline that binds a launch (the longer of its FLOPs at the bf16
    peak and its bytes at the HBM peak), the fraction of it reached, and both
    single-resource fractions."""
    t_f = flops / (peaks["bf16_tflops"] * 1e12)
    t_b = nbytes / (peaks["hbm_gbs"] * 1e9) if nbytes else 0.0
    t = ms * 1e-3
    return {"bound": "tensor" if t_f >= t_b else "hbm", "frac_roofline": round(max(t_f, t_b) / t, 4),
            "frac_bf16": round(t_f / t, 4), "frac_hbm": round(t_b / t, 4) if nbytes else None,
            "intensity_flop_per_byte": round(flops / nbytes, 1) if nbytes else None}


def build_prefill_launches(args, pka, device):
    import torch
    w = args.workload
    launches = []
    if w in ("encoder-prefill", "chunked-prefill", "t5-encoder-prefill"):
        if w == "chunked-prefill":
            layers = [synth.chunked_prefill_workload(device=device)]
        elif w == "t5-encoder-prefill":
            layers = [synth.t5_encoder_prefill_workload(device=device)]
        else:
            layers = [synth.prefill_workload(l, device=device, head_dim=getattr(args, "head_dim", 64))
                      for l in range(3)]
        cu = torch.from_numpy(layers[0].cu_seqlens).to(device)
        for c in layers:
            q, k, v = c.device_qkv
            out = torch.empty_like(q)
            if c.rel_bias is not None:
                rel = torch.from_numpy(c.rel_bias).to(device)
                fn = (lambda c=c, q=q, k=k, v=v, out=out, rel=rel:
                      pka.prefill_biased(out, q, k, v, cu, c.max_seqlen, rel, c.window, c.causal, c.scale))
            elif c.chunk > 0:
                fn = (lambda c=c, q=q, k=k, v=v, out=out:
                      pka.chunked_prefill(out, q, k, v, cu, c.max_seqlen, c.chunk, c.causal, c.scale))
            else:
                fn = (lambda c=c, q=q, k=k, v=v, out=out:
                      pka.swa_prefill(out, q, k, v, cu, c.max_seqlen, c.window, c.causal, c.scale))
            launches.append(PrefillLaunch(c.name, c, fn, out, prefill_flops(c), [q, k, v, cu],
                                          nbytes=packed_prefill_bytes(c)))
        return launches
    # t5-paged-prefill: a prompt chunk of every sequence of the T5-large decode
    # batch against the self-attention cache (its K/V written first) and the
    # encoder cross-attention cache
    self_c, cross_c = synth.t5_paged_prefill_workload(device=device)
    q = self_c.device_q
    cuq = torch.from_numpy(self_c.cu_seqlens_q).to(device)
    for pc in (self_c, cross_c):
        c = pc.cache
        H, D = c.num_heads, c.head_dim
        kc = torch.zeros((c.num_blocks, H, 16, D), dtype=torch.bfloat16, device=device)
        vc = torch.zeros_like(kc)
        key, value = c.device_kv
        pka.reshape_and_cache(key, value, kc, vc, torch.from_numpy(c.slot_mapping).to(device))
        bt = torch.from_numpy(np.ascontiguousarray(c.block_tables)).to(device)
        cl = torch.from_numpy(c.context_lens).to(device)
        rel = torch.from_numpy(pc.rel_bias).to(device) if pc.rel_bias is not None else None
        out = torch.empty_like(q)
        ins = [q, bt, cl, cuq] + ([rel] if rel is not None else [])
        pre = None
        if pc.causal:
            # the chunk's own K/V rows: the last Lq positions of each sequence
            qpos = np.concatenate([c.tok_offsets[s] + c.context_lens[s] - np.arange(l, 0, -1)
                                   for s, l in enumerate(pc.query_lens)]).astype(np.int64)
            idx = torch.from_numpy(qpos).to(device)
            new_k, new_v = key[idx].contiguous(), value[idx].contiguous()
            slots = torch.from_numpy(c.slot_mapping[qpos]).to(device)
            pre = (lambda new_k=new_k, new_v=new_v, kc=kc, vc=vc, slots=slots:
                   pka.reshape_and_cache(new_k, new_v, kc, vc, slots))
            ins += [new_k, new_v, slots]
        fn = (lambda pc=pc, out=out, kc=kc, vc=vc, bt=bt, cl=cl, rel=rel:
              pka.paged_prefill(out, q, kc, vc, bt, cuq, cl, pc.max_query_len, pc.window, pc.causal, rel, pc.scale))
        launches.append(PrefillLaunch(pc.name, pc, fn, out, 4 * D * H * pc.kept_pairs(), ins, pre,
                                      nbytes=paged_prefill_bytes(pc)))
        del key, value
        c.device_kv = None
    torch.cuda.empty_cache()
    return launches


def run_prefill(args, rank, world, local, peaks):
    import torch
    import paged_kv_attention_23_gb300 as pka
    pka.load()
    device = f"cuda:{local}"
    torch.cuda.set_device(local)
    launches = build_prefill_launches(args, pka, device)
    flops = [l.flops for l in launches]

    def step(events=None, k=0):
        for j, l in enumerate(launches):
            if l.pre is not None:
                l.pre()
            if events is not None:
                events[j][0][k].record()
            l.fn()
            if events is not None:
                events[j][1][k].record()

    clocks = ClockSampler(gpu_id(local))
    clocks.start()
    t_end = time.time() + args.clock_soak
    while time.time() < t_end:
        step(); torch.cuda.synchronize()
    for _ in range(args.warmup):
        step()
    K = args.steps
    graph = capture_graph(lambda: [step() for _ in range(K)])
    graph.replay()
    t0 = torch.cuda.Event(enable_timing=True); t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(); barrier(world)
    queue_ahead()
    t0.record()
    graph.replay()
    t1.record()
    torch.cuda.synchronize(); barrier(world)
    ms_step = max_over_ranks(t0.elapsed_time(t1), world) / K
    del graph
    # each call's launch time from a graph of K launches of that call alone
    launch_ms = [graph_ms(lambda k, l=l: l.fn(), K, world) for l in launches]
    clk = clocks.stop()
    pair_ms = per_launch_ms(lambda ev: [step(ev, k) for k in range(K)], len(launches), K)
    value = sum(flops) * world / (ms_step * 1e-3) / 1e12
    jd = int(np.argmax(flops))
    cases = [l.case for l in launches]
    bounds = [prefill_bound(l.flops, l.nbytes, m, peaks) for l, m in zip(launches, launch_ms)]
    packed = args.workload != "t5-paged-prefill"
    qkv_bytes = [4 * c.num_tokens * c.num_heads * c.head_dim * 2 for c in cases]
    kname = {"t5-paged-prefill": "paged_prefill (self-attention, causal + T5 bias)",
             "t5-encoder-prefill": "prefill_biased (T5 encoder layer)"}.get(args.workload,
                                                                         "swa_prefill (full-attention layer)")
    # the dominant launch against the roofline that binds it: the tensor peak
    # when its FLOPs take longer there than its bytes at the HBM peak, else HBM
    bd = bounds[jd]
    if bd["bound"] == "tensor":
        ach, peak, unit = flops[jd] / (launch_ms[jd] * 1e-3) / 1e12, peaks["bf16_tflops"], "TFLOP/s"
        peak_src = peaks["src"] + " bf16_tflops (burst)"
    else:
        ach, peak, unit = launches[jd].nbytes / (launch_ms[jd] * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s"
        peak_src = peaks["src"] + " hbm_gbs"
    traffic_key = args.workload + ("" if args.head_dim == 64 else f"-d{args.head_dim}")
    roof = {"bound": bd["bound"], "achieved": round(ach, 2), "peak": peak, "unit": unit,
            "frac": round(ach / peak, 4), "traffic": recorded_traffic("swa_prefill.cu", traffic_key),
            "kernel": kname, "alg_flops_per_launch": flops[jd], "alg_bytes_per_launch": launches[jd].nbytes,
            "frac_bf16": bd["frac_bf16"], "frac_hbm": bd["frac_hbm"],
            "intensity_flop_per_byte": bd["intensity_flop_per_byte"],
            "launch_ms": round(launch_ms[jd], 4), "launch_timing": "a graph of that launch alone / launches",
            "peak_src": peak_src}
    extra = {"launch_ms": [round(x, 4) for x in launch_ms],
             "launch_ms_event_pairs": [round(x, 4) for x in pair_ms],
             "launch_TFLOPs": [round(f / (m * 1e-3) / 1e12, 2) for f, m in zip(flops, launch_ms)],
             "launch_GBps": [round(l.nbytes / (m * 1e-3) / 1e9, 1) for l, m in zip(launches, launch_ms)],
             "launch_bounds": bounds,
             "flops_per_step": sum(flops)}
    if args.workload == "encoder-prefill":
        extra["window_layer_GBps"] = [round(b / (m * 1e-3) / 1e9, 1) for b, m in zip(qkv_bytes[1:], launch_ms[1:])]
        extra["window_layer_hbm_frac"] = [round(b / (m * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)
                                          for b, m in zip(qkv_bytes[1:], launch_ms[1:])]
    e2e = prefill_e2e(args, launches, sum(flops), world) if not args.no_e2e else None
    c0 = cases[0]
    cfg = {"workload": args.workload, "num_seqs": c0.num_seqs, "num_tokens": c0.num_tokens,
           "num_heads": c0.num_heads, "head_dim": c0.head_dim, "windows": [c.window for c in cases],
           "causal": [c.causal for c in cases], "parallelism": f"replicas x{world}"}
    if packed:
        cfg["chunks"] = [getattr(c, "chunk", 0) for c in cases]
        cfg["l2"] = f"q/k/v {qkv_bytes[0] * 3 / 4 / 2**20:.0f} MiB per layer > L2"
        cfg["bias"] = ["T5 relative-position table [H, 257] in kernel" if c.rel_bias is not None else None
                       for c in cases]
    else:
        cfg["context_lens"] = ["U[1,2048] (self)", "512 (cross)"]
        cfg["query_lens"] = "min(ctx, U[1,256])"
        cfg["bias"] = ["T5 table, non-negative half (self)", None]
        cfg["l2"] = "self + cross caches 1.6 GB > L2"
    res = {"value": value, "unit": "TFLOP/s", "ms_per_step": ms_step, "dtype": "bf16", "config": cfg,
           "roofline": roof, "e2e": e2e, "clocks": clk,
           "gpu_launches": K * sum(1 + (l.pre is not None) for l in launches), "extra": extra}
    if args.workload == "encoder-prefill" and args.per_config:
        res["record"] = prefill_record(launches, K, peaks, world, ms_step=ms_step, launch_ms=launch_ms)
    del launches
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def prefill_record(launches, K, peaks, world=1, ms_step=None, launch_ms=None):
    """Graph-timed layer launches and step of the encoder prefill: TFLOP/s and
    the fraction of the bf16 peak per layer and for the step; every layer also
    in GB/s of its algorithmic bytes (q, k, v read, out written) with the
    roofline that binds it."""
    if launch_ms is None:
        launch_ms = [graph_ms(lambda k, l=l: l.fn(), K, world) for l in launches]
    if ms_step is None:
        ms_step = graph_ms(lambda k: [l.fn() for l in launches], K, world)
    bf16, hbm = peaks["bf16_tflops"], peaks["hbm_gbs"]
    layers = []
    for l, ms in zip(launches, launch_ms):
        c = l.case
        tf = l.flops / (ms * 1e-3) / 1e12
        e = {"layer": c.name, "window": c.window, "ms_per_launch": round(ms, 4), "TFLOPs": round(tf, 1),
             "frac_bf16": round(tf / bf16, 4), "alg_flops": l.flops}
        if l.nbytes:
            e["GBps"] = round(l.nbytes / (ms * 1e-3) / 1e9, 1)
            e["frac_hbm"] = round(l.nbytes / (ms * 1e-3) / 1e9 / hbm, 4)
            e["alg_bytes"] = l.nbytes
            e["bound"] = prefill_bound(l.flops, l.nbytes, ms, peaks)["bound"]
        layers.append(e)
    flops = sum(l.flops for l in launches)
    tf = flops / (ms_step * 1e-3) / 1e12
    return {"layers": layers, "step": {"ms_per_step": round(ms_step, 4), "TFLOPs": round(tf, 1),
                                       "frac_bf16": round(tf / bf16, 4), "alg_flops": flops},
            "timing": "one CUDA graph of K launches per layer, and of K steps"}


def per_config_records(args, world, local, peaks, headline):
    """Every target workload measured the same way in the same run: decode
    configs graph-timed bias on and off (and, for the T5-large step, each
    attention type's own launch); the encoder prefill per layer and per step.
    The headline workload's record comes from its own run."""
    import torch
    import paged_kv_attention_23_gb300 as pka
    device = f"cuda:{local}"
    out = {}
    clocks = ClockSampler(gpu_id(local))
    clocks.start()
    for n, name in ((1, "tiny-decode"), (2, "t5-small-decode"), (3, "t5-large-decode"), (4, "encoder-prefill"),
                    (5, "long-ctx-decode")):
        key = f"config {n}: {name}"
        if name == args.workload and headline is not None:
            out[key] = headline
            continue
        if name == "encoder-prefill":
            launches = build_prefill_launches(argparse.Namespace(workload=name, head_dim=64), pka, device)
            for _ in range(args.warmup):
                for l in launches:
                    l()
            out[key] = prefill_record(launches, args.steps, peaks, world)
            del launches
        else:
            db = DecodeBench(name, pka, device)
            for w in range(args.warmup):
                db.step(w)
            out[key] = db.record(args.steps, peaks, world)
            del db
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    out["clocks"] = clocks.stop()
    return out


def prefill_e2e(args, launches, flops, world):
    """The same step through the public API from pinned host buffers: each
    call's inputs copied host->device, the call, its output read back.  The
    input copies run on a second stream and the read-backs on a third, ordered
    by events, so a layer's inputs arrive while the previous layer computes
    and outputs leave while later inputs arrive (as a serving engine pipelines
    a step; the host link carries both directions at once); every copy of a
    step is still inside the timed region."""
    import torch
    # Each distinct device input is copied once per step, in the batch of the
    # first call that reads it (several calls share cu_seqlens, or q); the
    # next step's copy of a batch waits for the last call that reads any of it.
    hosts = []
    h2d = 0
    first = {}
    last_reader = list(range(len(launches)))
    for j, l in enumerate(launches):
        hs = []
        for t in l.host_inputs:
            if t.data_ptr() in first:
                i = first[t.data_ptr()]
                last_reader[i] = max(last_reader[i], j)
                continue
            first[t.data_ptr()] = j
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            hs.append((h, t))
            h2d += t.numel() * t.element_size()
        hosts.append(hs)
    hout = [torch.empty(l.out.shape, dtype=l.out.dtype, pin_memory=True) for l in launches]
    d2h = sum(l.out.numel() * l.out.element_size() for l in launches)
    main = torch.cuda.current_stream()
    copies = torch.cuda.Stream()
    backs = torch.cuda.Stream()
    n = len(launches)
    ev = lambda: torch.cuda.Event()
    inputs_in = [ev() for _ in range(n)]           # layer l's inputs on the device
    computed = [ev() for _ in range(n)]            # layer l's call done (its inputs free, its output ready)
    read_back = [ev() for _ in range(n)]           # layer l's output copied out
    started = [False] * n

    def step():
        for j, (l, hs) in enumerate(zip(launches, hosts)):
            with torch.cuda.stream(copies):
                if started[last_reader[j]]:
                    copies.wait_event(computed[last_reader[j]])   # the previous step's calls have read them
                for h, d in hs:
                    d.copy_(h, non_blocking=True)
                inputs_in[j].record(copies)
        for j, (l, ho) in enumerate(zip(launches, hout)):
            main.wait_event(inputs_in[j])
            if started[j]:
                main.wait_event(read_back[j])            # the previous step's output has left
            l()
            computed[j].record(main)
            started[j] = True
            with torch.cuda.stream(backs):
                backs.wait_event(computed[j])
                ho.copy_(l.out, non_blocking=True)
                read_back[j].record(backs)
        main.wait_event(read_back[n - 1])

    for _ in range(args.warmup):
        step()
    a = torch.cuda.Event(enable_timing=True); b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(); barrier(world)
    a.record()
    copies.wait_event(a)                                   # no copy of the timed steps starts before a
    backs.wait_event(a)
    for _ in range(args.steps):
        step()
    for j in range(n):
        main.wait_event(read_back[j])
    b.record()
    torch.cuda.synchronize(); barrier(world)
    ms = max_over_ranks(a.elapsed_time(b), world) / args.steps
    return {"value": round(flops * world / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 4),
            "copies": "inputs on a second stream, read-backs on a third, overlapping the calls"}


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------
def _host_sub_decode(case, seqs):
    """Host arrays for a subset of sequences (token rows from the generator)."""
    if case.device_kv is None and len(seqs) == case.num_seqs:
        return case
    ks, vs = [], []
    for s in seqs:
        a, b = int(case.tok_offsets[s]), int(case.tok_offsets[s + 1])
        if case.device_kv is not None:
            ks.append(_host_storage(case.device_kv[0][a:b], case.dtype))
            vs.append(_host_storage(case.device_kv[1][a:b], case.dtype))
        else:
            ks.append(case.key[a:b]); vs.append(case.value[a:b])
    ctx = case.context_lens[seqs]
    pool, bt, slot, tok = synth._paged_layout(np.random.default_rng(0), ctx, case.block_size)
    return synth.DecodeCase(case.name, case.dtype, len(seqs), case.num_heads, case.head_dim, case.block_size, pool,
                            ctx.astype(np.int32), bt, slot, tok, case.q[seqs], np.concatenate(ks),
                            np.concatenate(vs), case.bias[seqs] if case.bias is not None else None, case.window,
                            case.scale)


def _host_storage(t, code):
    import torch
    t = t.detach().contiguous().cpu()
    return t.view(torch.int16).numpy().view(np.uint16) if code == BF16 else t.numpy()


def oracle_decode_sample(cases, budget_s: float, seed: int = 0):
    """Time the oracle on seeded random sequences of each case until about
    budget_s seconds of CPU work; returns (bytes, seconds, threads, desc)."""
    import oracle
    oracle.build()
    rng = np.random.default_rng(seed)
    threads = oracle.default_threads()
    total_b = 0
    total_s = 0.0
    nseq = 0
    c0 = cases[0]
    t_start = time.time()
    while time.time() - t_start < budget_s:
        for c in cases:
            k = min(c.num_seqs, 8)
            seqs = np.sort(rng.choice(c.num_seqs, size=k, replace=False))
            sub = _host_sub_decode(c, seqs)
            kc = np.zeros((sub.num_blocks, sub.num_heads, 16, sub.head_dim), dtype=sub.key.dtype)
            vc = np.zeros_like(kc)
            t = time.time()
            oracle.reshape_and_cache(kc, vc, sub.key, sub.value, sub.slot_mapping, 16)
            oracle.paged_decode(sub.q, kc, vc, sub.block_tables, sub.context_lens, sub.bias, sub.window, sub.scale,
                                16, sub.dtype, nthreads=threads)
            total_s += time.time() - t
            total_b += decode_alg_bytes(sub, True)["total"]
            nseq += k
    desc = (f"{nseq} sequences drawn at random (all heads) from the {c0.name} batch, "
            f"oracle scatter + fp64 paged decode, {total_s:.1f} s")
    return total_b, total_s, threads, desc


def oracle_prefill_sample(cases, budget_s: float, seed: int = 0):
    """Time the oracle on seeded random query rows (all heads) of each case
    until about budget_s seconds of CPU work; returns (flops, s, threads, desc)."""
    import oracle
    oracle.build()
    rng = np.random.default_rng(seed)
    threads = oracle.default_threads()
    host = []
    for c in cases:
        if isinstance(c, synth.PagedPrefillCase):
            cc = c.cache
            kc = np.zeros((cc.num_blocks, cc.num_heads, 16, cc.head_dim), dtype=cc.key.dtype)
            vc = np.zeros_like(kc)
            oracle.reshape_and_cache(kc, vc, cc.key, cc.value, cc.slot_mapping, 16)
            host.append((c.q, kc, vc))
        elif c.device_qkv is not None:
            host.append(tuple(_host_storage(t, BF16) for t in c.device_qkv))
        else:
            host.append((c.q, c.k, c.v))
    flops = 0
    secs = 0.0
    nrows = 0
    t_start = time.time()
    while time.time() - t_start < budget_s:
        for c, (q, k, v) in zip(cases, host):
            rows = np.sort(rng.choice(c.num_tokens, size=min(64, c.num_tokens), replace=False)).astype(np.int64)
            t = time.time()
            if isinstance(c, synth.PagedPrefillCase):
                oracle.paged_prefill(q, k, v, c.cache.block_tables, c.cu_seqlens_q, c.cache.context_lens, c.window,
                                     c.causal, c.scale, 16, BF16, rel_bias=c.rel_bias, rows=rows, nthreads=threads)
            elif c.chunk > 0:
                oracle.prefill_chunked(q, k, v, c.cu_seqlens, c.chunk, c.causal, c.scale, BF16, rows=rows,
                                       nthreads=threads)
            elif c.rel_bias is not None:
                oracle.prefill_biased(q, k, v, c.cu_seqlens, c.window, c.causal, c.scale, BF16, c.rel_bias, rows=rows,
                                      nthreads=threads)
            else:
                oracle.prefill(q, k, v, c.cu_seqlens, c.window, c.causal, c.scale, BF16, rows=rows,
                               nthreads=threads)
            secs += time.time() - t
            flops += 4 * c.head_dim * c.num_heads * _kept_keys(c, rows)
            nrows += len(rows)
    desc = (f"{nrows} query rows drawn at random over {len(cases)} call(s) of {cases[0].name} (all heads), "
            f"fp64 oracle, {secs:.1f} s")
    return flops, secs, threads, desc


def _kept_keys(c, rows):
    """Keys the mask keeps, summed over the listed query rows."""
    paged = isinstance(c, synth.PagedPrefillCase)
    cu = c.cu_seqlens_q if paged else c.cu_seqlens
    tot = 0
    for i in rows:
        b = int(np.searchsorted(cu, i, side="right") - 1)
        L = int(cu[b + 1] - cu[b]); r = int(i - cu[b])
        Lk = int(c.cache.context_lens[b]) if paged else L
        p = Lk - L + r
        chunk = 0 if paged else c.chunk
        if chunk > 0:
            lo = p // chunk * chunk
            hi = min(Lk - 1, lo + chunk - 1)
        elif c.window > 0:
            lo, hi = max(0, p - c.window + 1), min(Lk - 1, p + c.window - 1)
        else:
            lo, hi = 0, Lk - 1
        if c.causal:
            hi = min(hi, p)
        tot += max(0, hi - lo + 1)
    return tot


def host_prefill_cases(workload, small=False, head_dim=64):
    """Host-drawn cases of a prefill workload for the oracle (small: fewer
    sequences of the same shape for the large T5 workloads)."""
    if workload == "chunked-prefill":
        return [synth.chunked_prefill_workload()]
    if workload == "t5-encoder-prefill":
        return [synth.t5_encoder_prefill_workload(num_seqs=32 if small else 256)]
    if workload == "t5-paged-prefill":
        return list(synth.t5_paged_prefill_workload(num_seqs=32))
    return [synth.prefill_workload(l, head_dim=head_dim) for l in range(3)]


def host_decode_cases(workload):
    """Host-drawn cases of a decode workload for the oracle: the whole batch
    for the small workloads, 32 sequences of the same shapes (the first 32
    draws of the same laws) for the multi-GB ones."""
    n = DECODE_WORKLOADS[workload]
    if n in (3, 5):
        cases = [synth.decode_workload(n, num_seqs=32)] + ([synth.cross_workload(num_seqs=32)] if n == 3 else [])
        return cases, "32 sequences of the same shapes, drawn on the host"
    return [synth.decode_workload(n)], "the whole batch, drawn on the host"


def oracle_leg(workload, budget_s, head_dim=64):
    """The fp64 oracle timed on the host cores on a bounded sample of the
    workload: (value, unit, threads, sample description, seconds)."""
    if workload in PREFILL_WORKLOADS:
        cases = host_prefill_cases(workload, small=True, head_dim=head_dim)
        oracle_prefill_sample(cases, 0.5)             # warm-up: pages the arrays in
        f, s, th, desc = oracle_prefill_sample(cases, budget_s)
        if workload == "t5-paged-prefill" or workload == "t5-encoder-prefill":
            desc += " (32 sequences of the same shapes, drawn on the host)"
        return f / s / 1e12, "TFLOP/s", th, desc, s
    cases, note = host_decode_cases(workload)
    oracle_decode_sample(cases, 0.5)
    b, s, th, desc = oracle_decode_sample(cases, budget_s)
    return b / s / 1e9, "GB/s", th, f"{desc} ({note})", s


def cpu_baseline(args):
    """The oracle leg in a child process: no CUDA context, no torch threads,
    no clock sampler -- the same conditions as the reference arm -- so the two
    arms' oracle numbers agree on the same box."""
    load = os.getloadavg()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-leg", "--workload", args.workload,
           "--cpu-seconds", str(args.cpu_seconds), "--head-dim", str(args.head_dim)]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600 + 4 * args.cpu_seconds)
    if r.returncode != 0:
        raise RuntimeError(f"oracle leg failed: {r.stderr[-2000:]}")
    d = json.loads(r.stdout.strip().splitlines()[-1])
    d["conditions"] = (f"child process without a CUDA context, {d['cores']} oracle threads; host load average "
                       f"{load[0]:.2f} (1 min) before it started")
    return d


def oracle_leg_main(args):
    val, unit, th, desc, _ = oracle_leg(args.workload, args.cpu_seconds, args.head_dim)
    print(json.dumps({"value": round(val, 6), "unit": unit, "cores": th, "kind": "oracle", "sample": desc}),
          flush=True)


def run_reference(args, rank, world):
    """--impl reference: the fp64 CPU oracle, timed on the host cores on a
    bounded sample per step."""
    if rank != 0:
        return None
    per = max(0.25, args.ref_seconds / max(1, args.steps + args.warmup))
    load = os.getloadavg()
    val, unit, th, desc, s = oracle_leg(args.workload, per * args.steps, args.head_dim)
    line = {"metric": METRIC, "value": round(val, 6), "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(s * 1e3 / max(1, args.steps), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": ({"workload": args.workload} if args.head_dim == 64
                       else {"workload": args.workload, "head_dim": args.head_dim}), "impl": "reference",
            "cpu_baseline": {"value": round(val, 6), "unit": unit, "cores": th, "kind": "oracle", "sample": desc,
                             "conditions": f"{th} oracle threads; host load average {load[0]:.2f} (1 min) before"},
            "e2e": {"value": round(val, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    return line


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="pka", choices=["pka", "reference"])
    ap.add_argument("--workload", default="long-ctx-decode",
                    choices=sorted(DECODE_WORKLOADS) + list(PREFILL_WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--separate-launches", action="store_true",
                    help="decode workloads: reshape_and_cache launches, then one decode launch per attention type")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--t5-table", action="store_true",
                    help="T5-bias decode workloads: compute the bias in the kernel from its [H,129] table")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="profiling only: fewer sequences than the named decode workload")
    ap.add_argument("--clock-soak", type=float, default=1.5,
                    help="seconds of untimed steps while nvidia-smi samples clocks before the warm-up")
    ap.add_argument("--per-config", dest="per_config", action="store_true", default=None,
                    help="also measure every target workload (default with one GPU and the default step)")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false")
    ap.add_argument("--head-dim", type=int, default=64, choices=[64, 128],
                    help="encoder-prefill only: the head dim of its three layers")
    ap.add_argument("--oracle-leg", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.head_dim != 64 and args.workload != "encoder-prefill":
        ap.error("--head-dim applies to --workload encoder-prefill only")
    args.warmup = max(3, args.warmup)
    if args.oracle_leg:
        oracle_leg_main(args)
        return
    rank, world, local = dist_setup()
    if args.per_config is None:
        args.per_config = (world == 1 and not args.separate_launches and not args.t5_table
                           and args.num_seqs is None and args.head_dim == 64)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    peaks = measured_peaks()
    if args.workload in PREFILL_WORKLOADS:
        res = run_prefill(args, rank, world, local, peaks)
    else:
        res = run_decode(args, rank, world, local, peaks)
    if rank != 0:
        return
    per_cfg = per_config_records(args, world, local, peaks, res.get("record")) if args.per_config else None
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(args)
    line = {"metric": METRIC, "value": round(res["value"], 3), "unit": res["unit"], "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(res["ms_per_step"], 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": res["dtype"],
            "data": "synthetic (seeded)", "config": res["config"], "roofline": res["roofline"],
            "cpu_baseline": cpu, "e2e": res["e2e"], "gpu_launches": res["gpu_launches"], "clocks": res["clocks"],
            "extra": dict(res["extra"], per_config=per_cfg)}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
