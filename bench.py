#!/usr/bin/env python3
"""Benchmark of the grouped-query attention forward hot path on one GB300.

One step = one pass of the whole path on seeded synthetic inputs:
  * decode  : Llama3-70B-shaped GQA decode, B=1, H_q=64, H_kv=8, d=128,
              ctx 32768 -- split-KV kernel + log-sum-exp combine;
  * prefill : Llama3-70B-shaped causal GQA prefill, B=1, S=8192, H_q=64,
              H_kv=8, d=128.
``value`` is the decode leg's KV-cache throughput (GB/s of K and V bytes read,
inputs resident in HBM; rotating K/V copies, at least 1.5 GiB of them, so
that no step finds its inputs in L2); the prefill leg's TFLOP/s (causal FLOPs
only) is reported beside it under ``prefill``.  The other workloads of the
same family -- the tiny d = 32 decode, the ragged batch-8 decode and the 64K
causal prefill -- are timed under the same rules and reported under
``configs``, each with its roofline, its parity against the fp64 oracle and
the oracle's own time on the host cores.

Timing: the K steps of a workload are captured once in a CUDA graph (the same
C-ABI launches, programmatic dependent launches included) and replayed once
between CUDA events on the launching stream.  The GPU is kept busy right up to
the start event: a GPU left idle runs the first few hundred microseconds of
work measurably slower (20 decode steps read 26-29 us each instead of 24 us
after 0.3-1 s of idle, with the SM and memory clocks reading full speed), so
the clock sampler is started before the warm-up, and an untimed lead-in graph
of the same workload is queued between the opening synchronise and the start
event.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the fp64 CPU oracle on the host cores instead
(bounded samples of the same workloads).  Under torchrun (N > 1) every rank runs
an independent replica (the path has no cross-GPU exchange); the value is the
sum over ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode KV GB/s (% HBM peak); causal prefill TFLOPS (% bf16 peak)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
NOMINAL_HBM_GBS = 8000.0        # the ~8 TB/s the decode target is stated against
NOMINAL_BF16_TFLOPS = 2250.0    # GB300 dense bf16 datasheet figure
REPEATS = 5                     # extra replays of each timed graph for the median and the min


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return (float(j["hbm_gbs"]), float(j["bf16_tflops"]),
                float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), "measured")
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS, "fallback"


def _source_digest(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "gqa_attention_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _recorded_traffic(profile_name, files):
    """Per-launch DRAM bytes recorded from an ncu capture, if the kernel is unchanged since."""
    path = os.path.join(ROOT, "profiles", profile_name)
    try:
        text = open(path).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith(("traffic_bytes_per_launch", "source_digest")):
            k, v = line.split(":", 1)
            fields[k.strip().lstrip("- ")] = v.strip().strip("`")
    try:
        if fields.get("source_digest") != _source_digest(files):
            return None
        return float(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


DECODE_SOURCES = ["decode.cu", "common.cuh", "internal.h"]
PREFILL_SOURCES = ["prefill.cu", "tcgen05.cuh", "common.cuh", "internal.h"]


def cpu_model():
    """Host CPU model name (lscpu on Arm, /proc/cpuinfo elsewhere)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"gqa_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------- helpers ---
def max_over_ranks(values, dist, device):
    """Element-wise maximum of `values` over all ranks (identity when dist is None)."""
    import torch

    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_rate(world, units_per_rank, seconds_slowest):
    """Aggregate throughput: every rank's units over the slowest rank's time."""
    return world * units_per_rank / seconds_slowest


# Decode inputs rotate through copies of the cache so that a copy is read again
# only after at least ROTATION_BYTES of other cache reads (12 x the 126 MB L2).
# The decode sweep loads K/V evict-first in L2, which leaves the lines that a
# step prefetched at normal priority; with 3 copies (384 MiB) some of them were
# still in L2 when their copy came round again (measured 1.1 us faster per
# step than with 12 copies), so a shorter rotation would overstate the rate.
ROTATION_BYTES = 3 << 29


def n_copies(bytes_per_copy):
    return max(2, -(-ROTATION_BYTES // bytes_per_copy))


def causal_flops(d, H_q, B, rows):
    """4 d FLOPs per (query row, visible key, query head); causal row i sees i + 1 keys."""
    return 4.0 * d * H_q * B * float(sum(int(r) + 1 for r in rows))


class TimedGraph:
    """A captured workload: `steps` timed steps plus the untimed steps around them."""

    def __init__(self, graph, steps, e0=None, e1=None, lead=None):
        self.graph, self.steps, self.e0, self.e1, self.lead = graph, steps, e0, e1, lead


class GraphTimer:
    """Times K steps of a workload from one replay of a CUDA graph that holds them.

    The graph holds, in stream order, an untimed lead-in of the same workload
    (~0.3 ms of GPU time, on the cache copies that precede the timed ones in the
    rotation), the start event, the K timed steps, the end event and, for a
    decode, one untimed step after them.  The events are event-record nodes of
    the graph, so the timed steps start from the steady state of a continuously
    loaded GPU, not from an idle one, and the count of timed steps does not
    change the per-step figure.  Each replay is bracketed by a barrier and a
    device synchronise on both sides.  Where the installed torch cannot record
    events inside a graph, the lead-in is a graph of its own replayed just
    before the start event."""

    LEAD_MS = 0.3  # GPU time the lead-in covers

    def __init__(self, torch, stream, dist):
        self.torch = torch
        self.stream = stream
        self.dist = dist
        self.side = torch.cuda.Stream()
        try:
            torch.cuda.Event(enable_timing=True, external=True)
            self.inner_events = True
        except TypeError:
            self.inner_events = False

    def _event(self):
        if self.inner_events:
            return self.torch.cuda.Event(enable_timing=True, external=True)
        return self.torch.cuda.Event(enable_timing=True)

    def _capture(self, body):
        torch = self.torch
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        self.side.wait_stream(self.stream)
        with torch.cuda.graph(graph, stream=self.side):
            body(torch.cuda.current_stream())
        torch.cuda.synchronize()
        return graph

    def _estimate_ms(self, fn, start):
        """GPU ms per step of three eager steps (sizes the lead-in)."""
        torch = self.torch
        fn(start, self.stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for i in range(3):
            fn(start + i, self.stream)
        e1.record(self.stream)
        e1.synchronize()
        return max(e0.elapsed_time(e1) / 3, 1e-6)

    def prepare(self, fn, steps, copies=None, lead_out=0):
        """Capture fn(0..steps-1) as the timed steps; `copies` is the length of
        the workload's cache rotation (None: no rotation)."""
        n = max(1, math.ceil(self.LEAD_MS / self._estimate_ms(fn, 0)))
        start = 0
        if copies is not None:
            n = min(n, copies)
            start = copies - n
        if self.inner_events:
            e0, e1 = self._event(), self._event()

            def body(s):
                for i in range(n):
                    fn(start + i, s)
                e0.record(s)
                for i in range(steps):
                    fn(i, s)
                e1.record(s)
                for i in range(lead_out):
                    fn(steps + i, s)

            tg = TimedGraph(self._capture(body), steps, e0, e1)
        else:
            graph = self._capture(lambda s: [fn(i, s) for i in range(steps)])
            lead = self._capture(lambda s: [fn(start + i, s) for i in range(n)])
            tg = TimedGraph(graph, steps, lead=lead)
        self.warm(tg)
        return tg

    def warm(self, tg):
        if tg.lead is not None:
            tg.lead.replay()
        tg.graph.replay()
        self.torch.cuda.synchronize()

    def _barrier(self):
        if self.dist is not None:
            self.dist.barrier()
        self.torch.cuda.synchronize()

    def time(self, tg):
        """Mean ms per timed step of one replay."""
        torch = self.torch
        self._barrier()
        with torch.cuda.stream(self.stream):
            if tg.e0 is not None:
                tg.graph.replay()
                e0, e1 = tg.e0, tg.e1
            else:
                e0, e1 = self._event(), self._event()
                tg.lead.replay()
                e0.record(self.stream)
                tg.graph.replay()
                e1.record(self.stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        self._barrier()
        return ms / tg.steps

    def time_repeated(self, tg, repeats):
        """(first replay, [all replays]) in ms per step."""
        first = self.time(tg)
        return first, [first] + [self.time(tg) for _ in range(repeats)]


def _repeat_stats(ms_list):
    return {"n": len(ms_list), "median_ms": round(statistics.median(ms_list), 6),
            "min_ms": round(min(ms_list), 6), "max_ms": round(max(ms_list), 6)}


# ------------------------------------------------------------ workloads ---
class DecodeLeg:
    """A decode workload: split kernel (+ combine when split) over rotating cache copies."""

    def __init__(self, torch, g, cfg, dev, seed=0, balanced=False, n_split=None):
        from gqa_attention_gb300 import inputs

        self.torch, self.g, self.cfg, self.dev = torch, g, cfg, dev
        q, k, v, lens = inputs.decode_inputs_for(cfg, seed=seed)
        self.host = (q, k, v, lens)
        self.lens_host = lens
        self.kv_bytes = 4 * cfg.d * cfg.H_kv * int(lens.sum())
        self.copies = n_copies(self.kv_bytes)
        self.qd, self.ld = q.to(dev), lens.to(dev)
        kd, vd = k.to(dev), v.to(dev)
        # all copies in one allocation each for K and V (views per copy)
        self.kall = torch.empty((self.copies,) + tuple(k.shape), dtype=k.dtype, device=dev)
        self.vall = torch.empty_like(self.kall)
        self.kall.copy_(kd.unsqueeze(0).expand_as(self.kall))
        self.vall.copy_(vd.unsqueeze(0).expand_as(self.vall))
        del kd, vd
        self.n_split = (n_split if n_split is not None else
                        g.gqa_attn_decode_default_splits(cfg.B, cfg.H_kv, cfg.S_max, dev.index))
        self.ws = g.decode_workspace(cfg.B, cfg.H_q, cfg.d, self.n_split, dev)
        # balanced splits: the claim counters, zeroed once (every call leaves them at zero)
        self.counters = (g.decode_counters(cfg.B, cfg.H_kv, dev)
                         if balanced and self.n_split > 1 else None)
        self.out = torch.empty(cfg.B, cfg.H_q, cfg.d, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(cfg.B, cfg.H_q, dtype=torch.float32, device=dev)
        self.launches_per_step = 2 if self.n_split > 1 else 1
        self.ws_bytes = (g.gqa_attn_decode_workspace_bytes(cfg.B, cfg.H_q, cfg.d, self.n_split)
                         if self.n_split > 1 else 0)

    def split(self, i, stream):
        c, g = self.cfg, self.g
        j = i % self.copies
        if self.counters is not None:
            st = g.gqa_attn_decode_balanced(self.qd, self.kall[j], self.vall[j], self.ld, c.B,
                                            c.S_max, c.H_q, c.H_kv, c.d, c.scale, self.n_split,
                                            self.ws, self.counters, self.out, self.lse, stream)
        else:
            st = g.gqa_attn_decode(self.qd, self.kall[j], self.vall[j], self.ld, c.B, c.S_max,
                                   c.H_q, c.H_kv, c.d, c.scale, self.n_split, self.ws, self.out,
                                   self.lse, stream)
        if st:
            raise RuntimeError(f"decode failed: {g.status_str(st)}")

    def step(self, i, stream):
        # split kernel + combine kernel back to back (the combine may overlap the
        # split kernel's tail through programmatic dependent launch)
        self.split(i, stream)
        if self.n_split > 1:
            c, g = self.cfg, self.g
            st = g.gqa_attn_decode_combine(self.ws, c.B, c.H_q, c.d, self.n_split, self.out,
                                           self.lse, stream)
            if st:
                raise RuntimeError(f"combine failed: {g.status_str(st)}")

    def all_bytes(self):
        """Every byte the step moves: K/V, Q, the split partials written and read back, O, LSE."""
        c = self.cfg
        return (self.kv_bytes + c.B * c.H_q * c.d * 2 + 2 * self.ws_bytes
                + c.B * c.H_q * (c.d * 2 + 4))

    def results(self):
        return self.out.float().cpu(), self.lse.float().cpu()


class Fp8DecodeLeg(DecodeLeg):
    """The decode workload over an E4M3 cache with per-token scales: FP8 split
    kernel (three times the default split count) + combine, rotating cache copies."""

    def __init__(self, torch, g, cfg, dev, seed=0):
        from gqa_attention_gb300 import inputs

        self.torch, self.g, self.cfg, self.dev = torch, g, cfg, dev
        q, k8, v8, ks, vs, lens = inputs.decode_inputs_fp8(cfg.B, cfg.H_q, cfg.H_kv, cfg.d,
                                                           cfg.S_max, seed=seed, ragged=cfg.ragged)
        self.host = (q, k8, v8, ks, vs, lens)
        self.lens_host = lens
        # bytes the sweep must read: E4M3 codes + one fp32 scale per token, for K and V
        self.kv_bytes = 2 * int(lens.sum()) * (cfg.H_kv * cfg.d + 4)
        self.copies = n_copies(self.kv_bytes)
        self.qd, self.ld = q.to(dev), lens.to(dev)
        self.caches = []
        for t in (k8, v8, ks, vs):  # all copies in one allocation per tensor
            a = torch.empty((self.copies,) + tuple(t.shape), dtype=t.dtype, device=dev)
            a.copy_(t.to(dev).unsqueeze(0).expand_as(a))
            self.caches.append(a)
        self.n_split = 3 * g.gqa_attn_decode_default_splits(cfg.B, cfg.H_kv, cfg.S_max, dev.index)
        self.ws = g.decode_workspace(cfg.B, cfg.H_q, cfg.d, self.n_split, dev)
        self.out = torch.empty(cfg.B, cfg.H_q, cfg.d, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(cfg.B, cfg.H_q, dtype=torch.float32, device=dev)
        self.launches_per_step = 2 if self.n_split > 1 else 1
        self.ws_bytes = (g.gqa_attn_decode_workspace_bytes(cfg.B, cfg.H_q, cfg.d, self.n_split)
                         if self.n_split > 1 else 0)

    def split(self, i, stream):
        c, g = self.cfg, self.g
        j = i % self.copies
        kc, vc, ksc, vsc = (a[j] for a in self.caches)
        st = g.gqa_attn_decode_fp8(self.qd, kc, vc, ksc, vsc, self.ld, c.B, c.S_max, c.H_q,
                                   c.H_kv, c.d, c.scale, self.n_split, self.ws, self.out,
                                   self.lse, stream)
        if st:
            raise RuntimeError(f"FP8 decode failed: {g.status_str(st)}")


class PrefillLeg:
    """A causal prefill workload (inputs larger than L2, re-read every step)."""

    def __init__(self, torch, g, cfg, dev, seed=0):
        from gqa_attention_gb300 import inputs

        self.torch, self.g, self.cfg, self.dev = torch, g, cfg, dev
        q, k, v = inputs.prefill_inputs_for(cfg, seed=seed)
        self.host = (q, k, v)
        self.qd, self.kd, self.vd = q.to(dev), k.to(dev), v.to(dev)
        self.out = torch.empty_like(self.qd)
        self.lse = torch.empty(cfg.B, cfg.H_q, cfg.S, dtype=torch.float32, device=dev)
        self.flops = causal_flops(cfg.d, cfg.H_q, cfg.B, range(cfg.S))
        self.launches_per_step = 1
        # query rows the oracle checks (and times): the configuration's own
        # sample where it names one, else 512 seeded rows
        self.rows = inputs.sample_rows(cfg.S, cfg.oracle_rows or 512, seed=seed)

    def step(self, i, stream):
        c, g = self.cfg, self.g
        st = g.gqa_attn_prefill_causal(self.qd, self.kd, self.vd, c.B, c.S, c.H_q, c.H_kv, c.d,
                                       c.scale, self.out, self.lse, stream)
        if st:
            raise RuntimeError(f"prefill failed: {g.status_str(st)}")

    def results(self):
        r = self.rows.to(self.dev)
        return (self.out.index_select(1, r).float().cpu(),
                self.lse.index_select(2, r).float().cpu())


def _hbm_roofline(kernel, bytes_per_launch, ms, hbm_gbs, peak_kind, traffic):
    achieved = bytes_per_launch / (ms * 1e-3) / 1e9
    return {"kernel": kernel, "bound": "hbm", "achieved": round(achieved, 2), "peak": hbm_gbs,
            "unit": "GB/s", "frac": round(achieved / hbm_gbs, 4), "peak_kind": peak_kind,
            "frac_of_nominal_8TBs": round(achieved / NOMINAL_HBM_GBS, 4),
            "traffic": traffic, "algorithmic_bytes_per_launch": bytes_per_launch}


def _tensor_roofline(kernel, flops, ms, bf16_tf, bf16_tf_sus, peak_kind, traffic):
    tf = flops / (ms * 1e-3) / 1e12
    return {"kernel": kernel, "bound": "tensor", "achieved": round(tf, 2), "peak": bf16_tf,
            "unit": "TFLOP/s", "frac": round(tf / bf16_tf, 4), "peak_kind": peak_kind + " (burst)",
            "frac_of_sustained": round(tf / bf16_tf_sus, 4),
            "frac_of_nominal_2250TF": round(tf / NOMINAL_BF16_TFLOPS, 4),
            "traffic": traffic, "algorithmic_flops_per_launch": flops}


# ------------------------------------------------------------------- ours ---
def run_ours(args, rank, world, dist):
    import torch

    import gqa_attention_gb300 as g
    from gqa_attention_gb300 import inputs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    g.load()
    stream = torch.cuda.current_stream()
    hbm_gbs, bf16_tf, bf16_tf_sus, peak_kind = _peaks()
    K = args.steps
    want_decode = args.only in (None, "decode")
    want_prefill = args.only in (None, "prefill")
    want_configs = args.only is None and not args.no_configs

    # ---------------- workloads ----------------
    seed = args.seed
    dec = (DecodeLeg(torch, g, inputs.LLAMA70B_DECODE, dev, seed=seed, n_split=args.splits)
           if want_decode else None)
    pre = PrefillLeg(torch, g, inputs.LLAMA70B_PREFILL_8K, dev, seed=seed) if want_prefill else None
    extra = {}
    if want_configs:
        # (the power-heavy 64K prefill last: the compute-bound FP8 decode is
        # sensitive to the clocks a long prefill leaves behind)
        extra["decode_tiny"] = DecodeLeg(torch, g, inputs.TINY_DECODE, dev, seed=seed)
        # (the ragged batch through the balanced splits: 1.5% faster than fixed ones)
        extra["decode_ragged"] = DecodeLeg(torch, g, inputs.LLAMA70B_DECODE_RAGGED, dev,
                                           seed=seed, balanced=True)
        extra["decode_fp8"] = Fp8DecodeLeg(torch, g, inputs.LLAMA70B_DECODE, dev, seed=seed)
        extra["prefill_64k"] = PrefillLeg(torch, g, inputs.PREFILL_64K, dev, seed=seed)
    legs = [x for x in (dec, pre, *extra.values()) if x is not None]

    # one eager call of each workload (library set-up happens outside any capture)
    for leg in legs:
        leg.step(0, stream)
    torch.cuda.synchronize()
    if g.gqa_last_device_error(stream) != g.GQA_OK:
        raise RuntimeError("device error in the first calls")

    timer = GraphTimer(torch, stream, dist)
    graphs, split_graphs = {}, {}
    for leg in legs:
        dec_leg = isinstance(leg, DecodeLeg)
        copies = leg.copies if dec_leg else None
        graphs[id(leg)] = timer.prepare(leg.step, K, copies, lead_out=1 if dec_leg else 0)
        if dec_leg and leg.n_split > 1:
            split_graphs[id(leg)] = timer.prepare(leg.split, K, copies, lead_out=1)

    with ClockSampler(dev.index) as clk:
        t_wall = time.perf_counter()
        timed = {}
        for leg in legs:
            # warm-up right before this workload's timed regions: W steps, one
            # read of every rotating cache copy, one replay of its graphs
            for i in range(args.warmup):
                leg.step(i, stream)
            if isinstance(leg, DecodeLeg):
                for c in range(leg.copies):
                    leg.step(c, stream)
            timer.warm(graphs[id(leg)])
            if g.gqa_last_device_error(stream) != g.GQA_OK:
                raise RuntimeError("device error during warm-up")
            # timed regions: K steps each
            timed[id(leg)] = timer.time_repeated(graphs[id(leg)], REPEATS)
            if id(leg) in split_graphs:
                timer.warm(split_graphs[id(leg)])
                timed[("split", id(leg))] = timer.time_repeated(split_graphs[id(leg)], REPEATS)
        wall_s = time.perf_counter() - t_wall
    clocks = clk.summary()
    if g.gqa_last_device_error(stream) != g.GQA_OK:
        raise RuntimeError("device error during the timed regions")
    results = {id(leg): leg.results() for leg in legs}

    # ---------------- end to end through the C ABI from pinned host buffers -----
    e2e = None
    if dec is not None and args.only is None:
        q, k, v, lens = dec.host
        hq, hk, hv, hl = (x.pin_memory() for x in (q, k, v, lens))
        hout = torch.empty(dec.out.shape, dtype=dec.out.dtype).pin_memory()
        hlse = torch.empty(dec.lse.shape, dtype=dec.lse.dtype).pin_memory()
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hl))
        d2h = hout.numel() * hout.element_size() + hlse.numel() * hlse.element_size()

        def e2e_step():
            dec.qd.copy_(hq, non_blocking=True)
            dec.kall[0].copy_(hk, non_blocking=True)
            dec.vall[0].copy_(hv, non_blocking=True)
            dec.ld.copy_(hl, non_blocking=True)
            dec.step(0, stream)
            hout.copy_(dec.out, non_blocking=True)
            hlse.copy_(dec.lse, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        e2e_steps = max(3, min(K, 50))
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        e1.synchronize()
        e2e = {"ms": e0.elapsed_time(e1) / e2e_steps, "h2d": h2d, "d2h": d2h}

        # The same decode with the cache resident in HBM, as a serving step runs
        # it.  The step's inputs (the query, the lengths and the new token's K
        # and V rows, one per KV head) travel in one pinned staging buffer and
        # one host-to-device copy; the call reads q and seq_lens in place in the
        # device copy of that buffer, the two rows are written at position
        # seq_lens[b] - 1 of the cache copy the step reads, and O and LSE, which
        # the call writes into one device buffer, come back in one copy.
        c = dec.cfg
        last = [int(x) - 1 for x in lens]

        def carve(parts):  # 256-byte aligned offsets of the parts in one buffer
            offs, n = [], 0
            for t in parts:
                offs.append(n)
                n += (t.numel() * t.element_size() + 255) // 256 * 256
            return offs, n

        rows_k = torch.stack([k[b, t] for b, t in enumerate(last)])  # [B, H_kv, d]
        rows_v = torch.stack([v[b, t] for b, t in enumerate(last)])
        parts_in = [q, lens.to(torch.int32), rows_k, rows_v]
        offs_in, n_in = carve(parts_in)
        stage_h = torch.zeros(n_in, dtype=torch.uint8).pin_memory()
        for o, t in zip(offs_in, parts_in):
            stage_h[o:o + t.numel() * t.element_size()].copy_(t.contiguous().view(-1).view(torch.uint8))
        stage_d = torch.empty(n_in, dtype=torch.uint8, device=dev)

        def view_of(buf, off, like):
            return buf[off:off + like.numel() * like.element_size()].view(like.dtype).view(like.shape)

        q_s, l_s, k_s, v_s = (view_of(stage_d, o, t) for o, t in zip(offs_in, parts_in))
        offs_out, n_out = carve([dec.out, dec.lse])
        res_d = torch.empty(n_out, dtype=torch.uint8, device=dev)
        res_h = torch.empty(n_out, dtype=torch.uint8).pin_memory()
        out_r, lse_r = view_of(res_d, offs_out[0], dec.out), view_of(res_d, offs_out[1], dec.lse)

        def e2e_resident_step(i, s):
            j = i % dec.copies
            stage_d.copy_(stage_h, non_blocking=True)
            for b, t in enumerate(last):
                dec.kall[j][b, t].copy_(k_s[b], non_blocking=True)
                dec.vall[j][b, t].copy_(v_s[b], non_blocking=True)
            st = g.gqa_attn_decode(q_s, dec.kall[j], dec.vall[j], l_s, c.B, c.S_max, c.H_q,
                                   c.H_kv, c.d, c.scale, dec.n_split, dec.ws, out_r, lse_r, s)
            if st == g.GQA_OK and dec.n_split > 1:
                st = g.gqa_attn_decode_combine(dec.ws, c.B, c.H_q, c.d, dec.n_split, out_r, lse_r,
                                               s)
            if st:
                raise RuntimeError(f"decode failed: {g.status_str(st)}")
            res_h.copy_(res_d, non_blocking=True)

        # (the K steps in a CUDA graph, as for the device-timed figures: Python
        # enqueues the step's six calls more slowly than the GPU runs them)
        for i in range(dec.copies):
            e2e_resident_step(i, stream)
        torch.cuda.synchronize()
        tg_res = timer.prepare(e2e_resident_step, K, dec.copies, lead_out=1)
        timer.warm(tg_res)
        e2e["resident_ms"] = timer.time(tg_res)
        e2e["resident_h2d"] = n_in
        e2e["resident_d2h"] = n_out
        # the outputs that came back equal, bit for bit, those of the device-timed decode
        o_h = view_of(res_h, offs_out[0], dec.out.cpu())
        e2e["resident_same"] = bool(torch.equal(o_h.view(torch.int16),
                                                dec.out.cpu().view(torch.int16)))

    # ---------------- max over ranks ----------------
    keys = sorted(timed, key=str)
    flat = []
    for key in keys:
        first, allv = timed[key]
        flat += [first] + allv
    flat.append(e2e["ms"] if e2e else 0.0)
    flat.append(e2e["resident_ms"] if e2e else 0.0)
    flat = max_over_ranks(flat, dist, dev)
    pos = 0
    for key in keys:
        n = 1 + len(timed[key][1])
        timed[key] = (flat[pos], flat[pos + 1:pos + n])
        pos += n
    if e2e:
        e2e["ms"] = flat[pos]
        e2e["resident_ms"] = flat[pos + 1]
    if rank != 0:
        return None

    def leg_report(leg):
        first, allv = timed[id(leg)]
        rep = {"ms_per_step": round(first, 6), "repeats": _repeat_stats(allv),
               "launches_per_step": leg.launches_per_step}
        c = leg.cfg
        if isinstance(leg, DecodeLeg):
            gbs = whole_job_rate(world, leg.kv_bytes, first * 1e-3) / 1e9
            rep.update({"value": round(gbs, 2), "unit": "GB/s",
                        "frac_of_" + peak_kind + "_hbm": round(gbs / world / hbm_gbs, 4),
                        "frac_of_nominal_8TBs": round(gbs / world / NOMINAL_HBM_GBS, 4),
                        "B": c.B, "H_q": c.H_q, "H_kv": c.H_kv, "d": c.d, "S_max": c.S_max,
                        "seq_lens": [int(x) for x in leg.lens_host] if c.B > 1 else c.S_max,
                        "n_split": leg.n_split, "kv_bytes": leg.kv_bytes,
                        "all_bytes": leg.all_bytes(),
                        "all_bytes_GBs": round(leg.all_bytes() / (first * 1e-3) / 1e9, 2),
                        "l2": f"{leg.copies} rotating cache copies "
                              f"({leg.copies * leg.kv_bytes >> 20} MiB of K/V read)"})
            split_key = ("split", id(leg))
            if split_key in timed:
                s_first, s_all = timed[split_key]
                rep["ms_split_kernel"] = round(s_first, 6)
                rep["split_repeats"] = _repeat_stats(s_all)
                kern_ms = s_first
            else:
                kern_ms = first
            fp8 = isinstance(leg, Fp8DecodeLeg)
            profile = ("decode_fp8_llama70b_ctx32768.md" if fp8 else
                       "decode_split_llama70b_ctx32768.md")
            traffic = (_recorded_traffic(profile, DECODE_SOURCES)
                       if c is inputs.LLAMA70B_DECODE else None)
            rep["roofline"] = _hbm_roofline(
                "gqa_decode_split_kernel" + (" (E4M3 cache)" if fp8 else ""), leg.kv_bytes,
                kern_ms, hbm_gbs, peak_kind, traffic)
            if fp8:
                rep["dtype"] = "e4m3 cache with fp32 per-token scales, bf16 q/out"
            rep["entry"] = ("gqa_attn_decode_fp8" if fp8 else "gqa_attn_decode_balanced"
                            if getattr(leg, "counters", None) is not None else "gqa_attn_decode")
            if leg.n_split > 1:
                rep["entry"] += " + gqa_attn_decode_combine"
        else:
            tf = whole_job_rate(world, leg.flops, first * 1e-3) / 1e12
            rep.update({"value": round(tf, 2), "unit": "TFLOP/s",
                        "frac_of_" + peak_kind + "_bf16": round(tf / world / bf16_tf, 4),
                        "frac_of_nominal_2250TF": round(tf / world / NOMINAL_BF16_TFLOPS, 4),
                        "B": c.B, "S": c.S, "H_q": c.H_q, "H_kv": c.H_kv, "d": c.d,
                        "value_scale": c.value_scale, "causal_flops": leg.flops,
                        "l2": f"inputs {(leg.qd.numel() + 2 * leg.kd.numel()) * 2 >> 20} MiB "
                              "(> L2), read again every step"})
            traffic = (_recorded_traffic("prefill_causal_llama70b_s8192.md", PREFILL_SOURCES)
                       if c is inputs.LLAMA70B_PREFILL_8K else None)
            rep["roofline"] = _tensor_roofline("gqa_prefill_causal_kernel", leg.flops, first,
                                               bf16_tf, bf16_tf_sus, peak_kind, traffic)
        return rep

    reports = {}
    if dec is not None:
        reports["decode_llama70b"] = leg_report(dec)
    if pre is not None:
        reports["prefill_8k"] = leg_report(pre)
    for name, leg in extra.items():
        reports[name] = leg_report(leg)

    # launches of this library's kernels inside the timed regions (each region
    # is K steps; every graph is replayed 1 + REPEATS times)
    launches = 0
    for leg in legs:
        launches += (1 + REPEATS) * K * leg.launches_per_step
        if id(leg) in split_graphs:
            launches += (1 + REPEATS) * K

    dr = reports.get("decode_llama70b")
    pr = reports.get("prefill_8k")
    value = dr["value"] if dr else None
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round((dr["ms_per_step"] if dr else 0.0) + (pr["ms_per_step"] if pr else 0.0), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded torch.randn, rounded to bf16)",
        "config": {
            "workload": f"{inputs.LLAMA70B_DECODE.name} (value) + "
                        f"{inputs.LLAMA70B_PREFILL_8K.name} (prefill)",
            "decode": ({k: dr[k] for k in ("B", "H_q", "H_kv", "d", "n_split", "kv_bytes",
                                           "all_bytes", "all_bytes_GBs", "l2")}
                       | {"ctx": inputs.LLAMA70B_DECODE.S_max,
                          "ms_split_plus_combine": dr["ms_per_step"],
                          "ms_split_kernel": dr.get("ms_split_kernel"),
                          "step_median_ms": dr["repeats"]["median_ms"],
                          "step_min_ms": dr["repeats"]["min_ms"],
                          "hbm_frac_of_" + peak_kind: dr["frac_of_" + peak_kind + "_hbm"],
                          "hbm_frac_of_nominal_8TBs": dr["frac_of_nominal_8TBs"]}) if dr else None,
            "prefill": {k: pr[k] for k in ("B", "S", "H_q", "H_kv", "d")} if pr else None,
            "seed": args.seed,
            "l2": "decode: rotating K/V copies, a copy is read again only after >= 1.5 GiB "
                  "(12 x L2) of other cache reads; prefill inputs exceed L2",
            "timing": ("each workload: one CUDA graph holding an untimed lead-in of the same "
                       "workload (~0.3 ms), the start event, the K timed steps, the end event "
                       "(and one untimed decode step); replayed with a barrier + synchronize on "
                       "both sides, warmed right before; events on the launching stream; "
                       f"{REPEATS} more replays give the median and the min"),
            "events_inside_graph": timer.inner_events,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "clocks": clocks,
        "roofline": dr["roofline"] if dr else (pr["roofline"] if pr else None),
        "gpu_launches": launches,
        "wall_s_timed_regions": round(wall_s, 3),
    }
    if e2e:
        line["e2e"] = {"value": round(whole_job_rate(world, dec.kv_bytes, e2e["ms"] * 1e-3) / 1e9, 2),
                       "unit": "GB/s", "h2d_bytes_per_step": e2e["h2d"],
                       "d2h_bytes_per_step": e2e["d2h"], "ms_per_step": round(e2e["ms"], 4),
                       "path": "gqa_attn_decode + gqa_attn_decode_combine through the C ABI, "
                               "eager launches, pinned host buffers copied in and out every step"}
        line["e2e"]["resident_cache"] = {
            "value": round(whole_job_rate(world, dec.kv_bytes, e2e["resident_ms"] * 1e-3) / 1e9, 2),
            "unit": "GB/s", "ms_per_step": round(e2e["resident_ms"], 4),
            "h2d_bytes_per_step": e2e["resident_h2d"], "d2h_bytes_per_step": e2e["resident_d2h"],
            "outputs_equal_device_run": e2e["resident_same"],
            "path": "the same calls with the K/V cache resident in HBM (rotating copies); each "
                    "step copies in one pinned buffer holding the query, seq_lens and the new "
                    "token's K and V rows, writes the rows into the cache, and copies O and LSE "
                    "out in one copy; the K steps, copies included, replayed as one CUDA graph "
                    "between its events"}
    line["prefill"] = ({"value": pr["value"], "unit": "TFLOP/s", "ms": pr["ms_per_step"],
                        "causal_flops": pr["causal_flops"], "repeats": pr["repeats"],
                        "roofline": pr["roofline"]} if pr else None)
    if want_configs:
        line["configs"] = {
            "decode_tiny": reports["decode_tiny"] | {"workload": inputs.TINY_DECODE.name},
            "decode_llama70b": {"see": "value, config.decode, roofline",
                                "workload": inputs.LLAMA70B_DECODE.name},
            "decode_ragged": reports["decode_ragged"] | {"workload": inputs.LLAMA70B_DECODE_RAGGED.name},
            "prefill_8k": {"see": "prefill", "workload": inputs.LLAMA70B_PREFILL_8K.name},
            "prefill_64k": reports["prefill_64k"] | {"workload": inputs.PREFILL_64K.name},
            "decode_fp8": reports["decode_fp8"] | {"workload": inputs.LLAMA70B_DECODE.name
                                                   + " with an E4M3 cache (FP8 bytes)"},
        }
    # the oracle on the host cores (and the parity of every timed output
    # against it): a single-GPU figure, taken on rank 0 at N = 1
    if not args.no_cpu_baseline and world == 1:
        oracle_legs = {"decode_llama70b": dec, "prefill_8k": pre, **extra}
        cpu = cpu_baseline(oracle_legs, {id(l): results[id(l)] for l in legs})
        if "decode_llama70b" in cpu:
            line["cpu_baseline"] = cpu["decode_llama70b"]["cpu_baseline"]
            line["parity"] = cpu["decode_llama70b"]["parity"]
        if pr and "prefill_8k" in cpu:
            line["prefill"]["cpu_baseline"] = cpu["prefill_8k"]["cpu_baseline"]
            line["prefill"]["parity"] = cpu["prefill_8k"]["parity"]
        for name in ("decode_tiny", "decode_ragged", "prefill_64k", "decode_fp8"):
            if want_configs and name in cpu:
                line["configs"][name].update(cpu[name])
    else:
        line["cpu_baseline"] = None
    return line


# ------------------------------------------------------ CPU oracle baseline --
PARITY_BAR = {"max_dO": 2e-2, "mean_dO": 2e-3, "max_dLSE": 1e-3}


def _parity(out_gpu, lse_gpu, out_ref, lse_ref, what):
    import numpy as np

    o = np.asarray(out_gpu.numpy(), dtype=np.float64)
    l_ = np.asarray(lse_gpu.numpy(), dtype=np.float64)
    do, dl = np.abs(o - out_ref), np.abs(l_ - lse_ref)
    r = {"compared": what, "max_dO": float(do.max()), "mean_dO": float(do.mean()),
         "max_dLSE": float(dl.max()), "finite": bool(np.isfinite(o).all() and np.isfinite(l_).all())}
    r["pass"] = bool(r["finite"] and all(r[k] <= v for k, v in PARITY_BAR.items()))
    return r


def cpu_baseline(legs, results):
    """Time the fp64 oracle on the host cores on each workload (whole, or a stated
    row sample) and compare the GPU outputs of the timed regions with it."""
    import oracle

    oracle.build()
    cores = os.cpu_count() or 1
    model = cpu_model()
    out = {}
    for name, leg in legs.items():
        if leg is None:
            continue
        if isinstance(leg, DecodeLeg):
            if isinstance(leg, Fp8DecodeLeg):
                q, k8, v8, ks, vs, lens = leg.host

                def run(n):
                    return oracle.decode_fp8(q, k8, v8, ks, vs, lens, leg.cfg.scale, nthreads=n)
            else:
                q, k, v, lens = leg.host

                def run(n):
                    return oracle.decode(q, k, v, lens, leg.cfg.scale, nthreads=n)
            reps = 5 if leg.kv_bytes < (256 << 20) else 1
            times = []
            for _ in range(reps):
                t0 = time.perf_counter()
                ref_o, ref_l = run(cores)
                times.append(time.perf_counter() - t0)
            t = statistics.median(times)
            cb = {"value": round(leg.kv_bytes / t / 1e9, 4), "unit": "GB/s", "cores": cores,
                  "cpu": model, "kind": "oracle",
                  "sample": f"whole {leg.cfg.name} decode"
                            f"{' over the E4M3 cache' if isinstance(leg, Fp8DecodeLeg) else ''}"
                            " (every query head, every visible key), "
                            f"fp64, median of {reps} run(s), {t:.3f} s each"}
            if leg.kv_bytes < (256 << 20):  # the same sample on one core
                t0 = time.perf_counter()
                run(1)
                cb["value_1core"] = round(leg.kv_bytes / (time.perf_counter() - t0) / 1e9, 4)
            o_gpu, l_gpu = results[id(leg)]
            par = _parity(o_gpu, l_gpu, ref_o, ref_l, "every output row")
        else:
            q, k, v = leg.host
            rows = leg.rows
            t0 = time.perf_counter()
            ref_o, ref_l = oracle.prefill_causal_rows(q, k, v, leg.cfg.scale, rows=rows,
                                                      nthreads=cores)
            t = time.perf_counter() - t0
            fl = causal_flops(leg.cfg.d, leg.cfg.H_q, leg.cfg.B, rows.tolist())
            cb = {"value": round(fl / t / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
                  "cpu": model, "kind": "oracle",
                  "sample": f"{len(rows)} seeded query rows (rows 0 and S-1 included) x "
                            f"{leg.cfg.H_q} heads of {leg.cfg.name}, fp64, {t:.3f} s; the rate "
                            "counts the causal FLOPs of those rows only"}
            o_gpu, l_gpu = results[id(leg)]
            par = _parity(o_gpu, l_gpu, ref_o, ref_l, f"{len(rows)} sampled query rows x all heads")
        out[name] = {"cpu_baseline": cb, "parity": par}
        del ref_o, ref_l
    return out


def run_reference(args, rank, world):
    """The oracle as the reference arm: K timed steps of the whole decode workload on CPU."""
    if rank != 0:
        return None
    import oracle
    from gqa_attention_gb300 import inputs

    oracle.build()
    dc = inputs.LLAMA70B_DECODE
    q, k, v, lens = inputs.decode_inputs_for(dc, seed=args.seed)
    kv_bytes = 2 * int(lens.sum()) * dc.H_kv * dc.d * 2
    cores = os.cpu_count() or 1
    for _ in range(args.warmup):
        oracle.decode(q, k, v, lens, dc.scale, nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode(q, k, v, lens, dc.scale, nthreads=cores)
    dt = (time.perf_counter() - t0) / args.steps
    value = kv_bytes / dt / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded torch.randn, bf16)",
        "config": {"workload": f"{dc.name} (value)", "l2": "n/a (CPU)",
                   "parallelism": "CPU threads"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "cpu": cpu_model(), "kind": "oracle",
                         "sample": f"whole {dc.name} decode per step (fp64 oracle)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------- further workloads ---
WORKLOADS = ("decode_tiny", "decode_ragged", "decode_paged16", "decode_paged128", "decode_fp8",
             "decode_fp8_ragged", "decode_multi2", "decode_multi4", "decode_multi8", "decode_multi16",
             "decode_paged16_multi8", "decode_paged128_multi8", "prefill_64k", "prefill_window",
             "prefill_chunk", "prefill_d64", "prefill_d32", "decode_trace", "prefill_trace", "mma_rate",
             "decode_shapes")

# Serving shapes of the Llama3-70B heads (B sequences of S tokens) for the
# decode_shapes sweep of the default split count, fixed and balanced.
SERVING_SHAPES = ((4, 32768), (16, 8192), (64, 4096), (16, 32768), (64, 8192), (2, 131072),
                  (32, 2048), (128, 1024))


def run_decode_shapes(args):
    """Decode step (split + combine) of each serving shape with the library's default
    split count, through gqa_attn_decode and gqa_attn_decode_balanced: K steps in a
    CUDA graph over rotating cache copies (>= 1.5 GiB), median of 5 replays.  The
    inputs are drawn on the device from a seeded generator (a throughput sweep: the
    kernels' parity is the tests' job)."""
    import torch

    import gqa_attention_gb300 as g
    from gqa_attention_gb300 import inputs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    g.load()
    stream = torch.cuda.current_stream()
    hbm_gbs, _, _, peak_kind = _peaks()
    timer = GraphTimer(torch, stream, None)
    gen = torch.Generator(device=dev).manual_seed(args.seed)
    cfg = inputs.LLAMA70B_DECODE
    H_q, H_kv, d, scale = cfg.H_q, cfg.H_kv, cfg.d, cfg.scale
    steps = max(1, args.steps)
    shapes = {}
    for B, S in SERVING_SHAPES:
        kv_bytes = 4 * d * H_kv * B * S
        copies = n_copies(kv_bytes)
        q = torch.randn(B, H_q, d, device=dev, generator=gen).to(torch.bfloat16)
        ks = [torch.randn(B, S, H_kv, d, device=dev, generator=gen).to(torch.bfloat16)
              for _ in range(copies)]
        vs = [torch.randn(B, S, H_kv, d, device=dev, generator=gen).to(torch.bfloat16)
              for _ in range(copies)]
        lens = torch.full((B,), S, dtype=torch.int32, device=dev)
        n = g.gqa_attn_decode_default_splits(B, H_kv, S, dev.index)
        ws = g.decode_workspace(B, H_q, d, n, dev)
        ctr = g.decode_counters(B, H_kv, dev)
        out = torch.empty(B, H_q, d, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(B, H_q, dtype=torch.float32, device=dev)
        row = {"B": B, "S": S, "n_split": n, "kv_bytes": kv_bytes, "copies": copies}
        for mode in ("fixed", "balanced"):
            if mode == "balanced" and n < 2:
                continue

            def step(i, s, mode=mode):
                j = i % copies
                if mode == "fixed":
                    st = g.gqa_attn_decode(q, ks[j], vs[j], lens, B, S, H_q, H_kv, d, scale, n,
                                           ws, out, lse, s)
                else:
                    st = g.gqa_attn_decode_balanced(q, ks[j], vs[j], lens, B, S, H_q, H_kv, d,
                                                    scale, n, ws, ctr, out, lse, s)
                if st == g.GQA_OK and n > 1:
                    st = g.gqa_attn_decode_combine(ws, B, H_q, d, n, out, lse, s)
                if st:
                    raise RuntimeError(f"decode failed: {g.status_str(st)}")

            for i in range(copies):
                step(i, stream)
            torch.cuda.synchronize()
            tg = timer.prepare(step, steps, copies, lead_out=1)
            timer.warm(tg)
            ms = statistics.median(timer.time(tg) for _ in range(REPEATS))
            gbs = kv_bytes / (ms * 1e-3) / 1e9
            row[mode] = {"us_per_step": round(ms * 1e3, 2), "GBs": round(gbs, 1),
                         "frac_of_" + peak_kind + "_hbm": round(gbs / hbm_gbs, 4)}
        if g.gqa_last_device_error(stream) != g.GQA_OK or not bool(torch.isfinite(out.float()).all()):
            raise RuntimeError(f"decode B={B} S={S}: device error or non-finite output")
        shapes[f"B{B}_S{S}"] = row
        del ks, vs
        torch.cuda.empty_cache()
    return {"metric": "decode KV GB/s over serving shapes (Llama3-70B heads, default splits)",
            "unit": "GB/s", "steps": steps, "shapes": shapes, "dtype": "bf16",
            "data": "synthetic (seeded device generator)",
            "timing": "K steps in a CUDA graph over rotating copies, median of 5 replays"}


def _shuffled_pages(k, v, page_size, seed):
    """Scatter a contiguous cache [B, S, H, d] into a pool of pages in a seeded random order."""
    import torch

    B, S, H, d = k.shape
    nb = -(-S // page_size)
    perm = torch.randperm(B * nb, generator=torch.Generator().manual_seed(seed))
    kp = torch.zeros(B * nb, page_size, H, d, dtype=k.dtype)
    vp = torch.zeros_like(kp)
    table = torch.zeros(B, nb, dtype=torch.int32)
    for b in range(B):
        for j in range(nb):
            p = int(perm[b * nb + j])
            lo, hi = j * page_size, min(S, (j + 1) * page_size)
            kp[p, : hi - lo] = k[b, lo:hi]
            vp[p, : hi - lo] = v[b, lo:hi]
            table[b, j] = p
    return kp, vp, table


def run_decode_trace(args):
    """Where the decode split kernel's time goes, from the trace build
    (-DGQA_TRACE=1): per-phase cycles per tile and the CTA timeline of the
    second of two back-to-back decode steps (bf16 at the default split count,
    FP8 at three times it).  A diagnostic, not a timing."""
    import numpy as np
    import torch

    from gqa_attention_gb300 import inputs

    g = _trace_build()
    dev = torch.device("cuda", torch.cuda.current_device())
    cfg = inputs.LLAMA70B_DECODE
    n19 = g.gqa_attn_decode_default_splits(cfg.B, cfg.H_kv, cfg.S_max, dev.index)
    out = {"metric": "decode split-kernel trace (diagnostic build, not a timing)",
           "workload": cfg.name, "units": "cycles per 64-token tile and consumer warp; "
           "timeline in us from the first CTA's entry"}
    for kind, n in (("bf16", n19), ("fp8", 3 * n19)):
        if kind == "fp8":
            host = inputs.decode_inputs_fp8(cfg.B, cfg.H_q, cfg.H_kv, cfg.d, cfg.S_max, seed=0)
            call = g.decode_fp8
        else:
            host = inputs.decode_inputs_for(cfg, seed=0)
            call = g.decode
        a = [x.to(dev) for x in host]
        for _ in range(max(3, args.warmup)):
            call(*a, n_split=n)
        torch.cuda.synchronize()
        assert g.gqa_trace_clear() == g.GQA_OK
        call(*a, n_split=n)
        call(*a, n_split=n)
        torch.cuda.synchronize()
        ctas = n * cfg.H_kv
        buf = np.zeros(ctas * 64, dtype=np.uint64)
        assert g.gqa_trace_read(buf, buf.nbytes) == g.GQA_OK
        rec = buf.reshape(ctas, 64).astype(np.float64)
        warps = rec[:, 8:56].reshape(ctas, 8, 6)
        used = warps[warps[:, :, 4] > 0]
        tiles = used[:, 5].sum()
        phases = {k: round(float(used[:, j].sum() / tiles), 1)
                  for j, k in enumerate(("wait", "qk", "softmax", "pv", "loop"))}
        t0 = rec[:, 0].min()
        rel = (rec[:, :5] - t0) / 1e3

        def pct(x):
            return [round(float(np.percentile(x, q)), 2) for q in (0, 50, 100)]

        out[f"{kind}_{n}_splits"] = {
            "per_tile": phases,
            "epilogue_cycles_median": {k: float(np.median(rec[:, 56 + j]))
                                       for j, k in enumerate(("warp_rendezvous", "partials_to_smem",
                                                              "merge_and_store"))},
            "prologue_cycles_median": {k: float(np.median(rec[:, 59 + j]))
                                       for j, k in enumerate(("seq_len_read", "length_checks",
                                                              "query_fragments"))},
            "timeline_us_min_median_max": {
                "entry": pct(rel[:, 0]), "release": pct(rel[:, 1]), "loop_start": pct(rel[:, 2]),
                "loop_end": pct(rel[:, 3]), "epilogue_end": pct(rel[:, 4]),
                "loop": pct(rel[:, 3] - rel[:, 2]), "epilogue": pct(rel[:, 4] - rel[:, 3])}}
    return out


def _trace_build():
    """Build the diagnostic (-DGQA_TRACE=1) library beside the default one and load it."""
    import torch

    import gqa_attention_gb300 as g
    from gqa_attention_gb300 import build

    pkg = os.path.join(ROOT, "gqa_attention_gb300")
    path = build.build(extra_flags=["-DGQA_TRACE=1"],
                       lib_path=os.path.join(pkg, "_build_trace", "libgqa_attn_trace.so"),
                       build_dir=os.path.join(pkg, "_build_trace", "obj"))
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    g.load(path)
    return g


def run_prefill_trace(args):
    """Where a causal prefill step's cycles go, from the trace build: medians
    over the recorded (CTA, head, tile) stamps of the Llama3-70B-shaped 8K
    prefill (second of two launches).  A diagnostic, not a timing."""
    import numpy as np
    import torch

    from gqa_attention_gb300 import inputs

    g = _trace_build()
    dev = torch.device("cuda", torch.cuda.current_device())
    cfg = inputs.LLAMA70B_PREFILL_8K
    q, k, v = (x.to(dev) for x in inputs.prefill_inputs_for(cfg, seed=0))
    for _ in range(max(3, args.warmup)):
        g.prefill_causal(q, k, v)
    torch.cuda.synchronize()
    assert g.gqa_trace_clear() == g.GQA_OK
    g.prefill_causal(q, k, v)
    torch.cuda.synchronize()
    buf = np.zeros(8 * 2 * 64 * 16, dtype=np.uint64)
    assert g.gqa_trace_prefill_read(buf, buf.nbytes) == g.GQA_OK
    t = buf.reshape(8, 2, 64, 16).astype(np.float64)

    def med(f):
        vals = [f(c, x, j) for c in range(8) for x in range(2) for j in range(4, 60)
                if t[c, x, j + 1, 0] > 0 and t[c, x, j, 14] > 0]
        return round(float(np.median(vals)), 0) if vals else None

    return {
        "metric": "causal prefill pipeline trace (diagnostic build, not a timing)",
        "workload": cfg.name, "units": "SM cycles, medians over CTAs 0-7, both heads, tiles 4-59",
        "head_period": med(lambda c, x, j: t[c, x, j + 1, 0] - t[c, x, j, 0]),
        "softmax_quarter0": {
            "s_to_registers": med(lambda c, x, j: t[c, x, j, 8] - t[c, x, j, 0]),
            "row_max": med(lambda c, x, j: t[c, x, j, 9] - t[c, x, j, 8]),
            "exponentials_and_p_stores": med(lambda c, x, j: t[c, x, j, 10] - t[c, x, j, 9]),
            "to_release": med(lambda c, x, j: t[c, x, j, 4] - t[c, x, j, 10])},
        "softmax_slowest_quarter": med(lambda c, x, j: max(t[c, x, j, 4:8]) - min(t[c, x, j, 0:4])),
        "last_release_to_mma_passing_wait": med(lambda c, x, j: t[c, x, j, 12] - max(t[c, x, j, 4:8])),
        "mma_wait_started_after_last_release": med(lambda c, x, j: t[c, x, j, 11] - max(t[c, x, j, 4:8])),
        "issue_pv": med(lambda c, x, j: t[c, x, j, 13] - t[c, x, j, 12]),
        "issue_next_s": med(lambda c, x, j: t[c, x, j, 14] - t[c, x, j, 13]),
        "next_s_issued_to_softmax_sees_it": med(lambda c, x, j: min(t[c, x, j + 1, 0:4]) - t[c, x, j, 14]),
        "mma_head_b_done_to_v_wait": med(lambda c, x, j: t[c, 0, j + 1, 15] - t[c, 1, j, 14]),
        "head_b_offset": med(lambda c, x, j: t[c, 1, j, 0] - t[c, 0, j, 0]),
    }


def run_mma_rate(args):
    """Cycles per tcgen05.mma of each operand form the tensor-core kernels use
    (trace build; one CTA per SM, zero operands), against the nominal 8192
    bf16 FLOP per clock per SM.  A diagnostic, not a timing of the path."""
    g = _trace_build()
    forms = ((0, "SS N=128", 64), (1, "TS N=128", 64), (2, "SS N=256", 128), (3, "SS N=64", 32),
             (4, "TS N=128, B MN-major (P V)", 64), (5, "prefill head step: 8 SS + 8 TS", 64))
    out = {"metric": "tcgen05.mma issue rate (diagnostic build, not a timing)",
           "units": "SM cycles per instruction, median over SMs; M = 128, K = 16, bf16 -> fp32",
           "iters": 512, "forms": {}}
    for form, name, nominal in forms:
        st, cyc = g.gqa_trace_mma_rate(form, 512)
        if st != g.GQA_OK:
            raise RuntimeError(f"gqa_trace_mma_rate({form}) -> {g.status_str(st)}")
        out["forms"][name] = {"cycles": round(cyc, 1), "nominal": nominal,
                              "fraction_of_nominal": round(nominal / cyc, 3)}
    return out


def run_workload(name, args):
    """One JSON line for a workload other than the headline step (same timing rules)."""
    import torch

    import gqa_attention_gb300 as g
    from gqa_attention_gb300 import inputs

    if name == "decode_trace":
        return run_decode_trace(args)
    if name == "mma_rate":
        return run_mma_rate(args)
    if name == "decode_shapes":
        return run_decode_shapes(args)
    if name == "prefill_trace":
        return run_prefill_trace(args)
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    g.load()
    stream = torch.cuda.current_stream()
    hbm_gbs, bf16_tf, _, peak_kind = _peaks()
    steps = max(1, args.steps)
    timer = GraphTimer(torch, stream, None)

    def timed(fn, copies=None):
        fn(0, stream)
        torch.cuda.synchronize()
        tg = timer.prepare(fn, steps, copies, lead_out=1 if copies is not None else 0)
        for i in range(max(3, args.warmup)):
            fn(i, stream)
        timer.warm(tg)
        first, allv = timer.time_repeated(tg, REPEATS)
        if g.gqa_last_device_error(stream) != g.GQA_OK:
            raise RuntimeError("device error")
        return first, _repeat_stats(allv)

    if name in ("decode_tiny", "decode_ragged"):
        cfg = inputs.TINY_DECODE if name == "decode_tiny" else inputs.LLAMA70B_DECODE_RAGGED
        leg = DecodeLeg(torch, g, cfg, dev, balanced=name == "decode_ragged")
        for c in range(leg.copies):
            leg.step(c, stream)
        ms, rep = timed(leg.step, leg.copies)
        gbs = leg.kv_bytes / (ms * 1e-3) / 1e9
        return {"metric": f"decode KV GB/s ({cfg.name})", "value": round(gbs, 2), "unit": "GB/s",
                "ms_per_step": round(ms, 5), "repeats": rep, "steps": steps,
                "n_split": leg.n_split, "kv_bytes": leg.kv_bytes,
                "frac_of_" + peak_kind + "_hbm": round(gbs / hbm_gbs, 4),
                "l2": f"{leg.copies} rotating K/V copies", "dtype": "bf16", "data": "synthetic"}

    if name.startswith("decode_fp8"):
        cfg = inputs.LLAMA70B_DECODE if name == "decode_fp8" else inputs.LLAMA70B_DECODE_RAGGED
        q, k8, v8, ks, vs, lens = inputs.decode_inputs_fp8(cfg.B, cfg.H_q, cfg.H_kv, cfg.d,
                                                           cfg.S_max, seed=0, ragged=cfg.ragged)
        # bytes the sweep must read: E4M3 codes + one fp32 scale per token, for K and V
        kv_bytes = 2 * int(lens.sum()) * (cfg.H_kv * cfg.d + 4)
        copies = n_copies(kv_bytes)
        qd, ld = q.to(dev), lens.to(dev)
        caches = [tuple(x.to(dev) for x in (k8, v8, ks, vs)) for _ in range(copies)]
        n = 3 * g.gqa_attn_decode_default_splits(cfg.B, cfg.H_kv, cfg.S_max, dev.index)
        ws = g.decode_workspace(cfg.B, cfg.H_q, cfg.d, n, dev)
        out = torch.empty(cfg.B, cfg.H_q, cfg.d, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(cfg.B, cfg.H_q, dtype=torch.float32, device=dev)

        def fstep(i, s):
            kc, vc, ksc, vsc = caches[i % copies]
            assert g.gqa_attn_decode_fp8(qd, kc, vc, ksc, vsc, ld, cfg.B, cfg.S_max, cfg.H_q,
                                         cfg.H_kv, cfg.d, cfg.scale, n, ws, out, lse,
                                         s) == g.GQA_OK
            assert g.gqa_attn_decode_combine(ws, cfg.B, cfg.H_q, cfg.d, n, out, lse,
                                             s) == g.GQA_OK

        for c in range(copies):
            fstep(c, stream)
        ms, rep = timed(fstep, copies)
        gbs = kv_bytes / (ms * 1e-3) / 1e9
        bf16_equiv = 2 * int(lens.sum()) * cfg.H_kv * cfg.d * 2
        return {"metric": f"FP8-cache decode GB/s ({cfg.name})", "value": round(gbs, 2),
                "unit": "GB/s", "ms_per_step": round(ms, 5), "repeats": rep, "steps": steps,
                "n_split": n, "fp8_bytes": kv_bytes,
                "bf16_equivalent_GBs": round(bf16_equiv / (ms * 1e-3) / 1e9, 2),
                "frac_of_" + peak_kind + "_hbm": round(gbs / hbm_gbs, 4),
                "l2": f"{copies} rotating cache copies",
                "dtype": "e4m3 cache, bf16 q/out", "data": "synthetic"}

    if name.startswith("decode_multi"):
        # T_q query tokens ending a Llama3-70B 32K cache (speculative verification):
        # the multi-token decode, and the chunked prefill on the same problem
        cfg = inputs.LLAMA70B_DECODE
        T_q = int(name[len("decode_multi"):])
        gen = torch.Generator().manual_seed(0)
        q = torch.randn(cfg.B, T_q, cfg.H_q, cfg.d, generator=gen).to(torch.bfloat16)
        k = torch.randn(cfg.B, cfg.S_max, cfg.H_kv, cfg.d, generator=gen).to(torch.bfloat16)
        v = torch.randn(cfg.B, cfg.S_max, cfg.H_kv, cfg.d, generator=gen).to(torch.bfloat16)
        lens = torch.full((cfg.B,), cfg.S_max, dtype=torch.int32)
        kv_bytes = 2 * int(lens.sum()) * cfg.H_kv * cfg.d * 2
        qd, ld = q.to(dev), lens.to(dev)
        nc = n_copies(kv_bytes)
        kds = [k.to(dev) for _ in range(nc)]
        vds = [v.to(dev) for _ in range(nc)]
        n = g.gqa_attn_decode_multi_default_splits(cfg.B, T_q, cfg.H_q, cfg.H_kv, cfg.S_max,
                                                   cfg.d)
        ws = g.decode_workspace(cfg.B * T_q, cfg.H_q, cfg.d, n, dev)
        out = torch.empty(cfg.B, T_q, cfg.H_q, cfg.d, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(cfg.B, T_q, cfg.H_q, dtype=torch.float32, device=dev)
        lse_c = torch.empty(cfg.B, cfg.H_q, T_q, dtype=torch.float32, device=dev)

        def mstep(i, s):
            assert g.gqa_attn_decode_multi(qd, kds[i % nc], vds[i % nc], ld, cfg.B, T_q, cfg.S_max,
                                           cfg.H_q, cfg.H_kv, cfg.d, cfg.scale, n, ws, out, lse,
                                           s) == g.GQA_OK
            assert g.gqa_attn_decode_combine(ws, cfg.B * T_q, cfg.H_q, cfg.d, n, out, lse,
                                             s) == g.GQA_OK

        def cstep(i, s):
            assert g.gqa_attn_prefill_chunk(qd, kds[i % nc], vds[i % nc], ld, cfg.B, T_q, cfg.S_max,
                                            cfg.H_q, cfg.H_kv, cfg.d, cfg.scale, -1, out, lse_c,
                                            s) == g.GQA_OK

        for c in range(nc):
            mstep(c, stream)
        ms, rep = timed(mstep, nc)
        ms_chunk, _ = timed(cstep, nc)
        gbs = kv_bytes / (ms * 1e-3) / 1e9
        return {"metric": f"multi-token decode KV GB/s ({cfg.name}, T_q={T_q})",
                "value": round(gbs, 2),
                "unit": "GB/s", "ms_per_step": round(ms, 5), "repeats": rep, "steps": steps,
                "n_split": n, "kv_bytes": kv_bytes,
                "frac_of_" + peak_kind + "_hbm": round(gbs / hbm_gbs, 4),
                "chunked_prefill_ms_same_problem": round(ms_chunk, 5),
                "l2": f"{nc} rotating K/V copies", "dtype": "bf16", "data": "synthetic"}

    if name.startswith("decode_paged") and "_multi" in name:
        # T_q query tokens ending a Llama3-70B 32K cache held in shuffled pages
        cfg = inputs.LLAMA70B_DECODE
        page = int(name[len("decode_paged"):name.index("_multi")])
        T_q = int(name[name.index("_multi") + len("_multi"):])
        gen = torch.Generator().manual_seed(0)
        q = torch.randn(cfg.B, T_q, cfg.H_q, cfg.d, generator=gen).to(torch.bfloat16)
        k = torch.randn(cfg.B, cfg.S_max, cfg.H_kv, cfg.d, generator=gen).to(torch.bfloat16)
        v = torch.randn(cfg.B, cfg.S_max, cfg.H_kv, cfg.d, generator=gen).to(torch.bfloat16)
        lens = torch.full((cfg.B,), cfg.S_max, dtype=torch.int32)
        kv_bytes = 2 * int(lens.sum()) * cfg.H_kv * cfg.d * 2
        kp, vp, table = _shuffled_pages(k, v, page, seed=0)
        qd, ld, td = q.to(dev), lens.to(dev), table.to(dev)
        nc = n_copies(kv_bytes)
        kps = [kp.to(dev) for _ in range(nc)]
        vps = [vp.to(dev) for _ in range(nc)]
        n = g.gqa_attn_decode_multi_default_splits(cfg.B, T_q, cfg.H_q, cfg.H_kv, cfg.S_max,
                                                   cfg.d)
        ws = g.decode_workspace(cfg.B * T_q, cfg.H_q, cfg.d, n, dev)
        out = torch.empty(cfg.B, T_q, cfg.H_q, cfg.d, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(cfg.B, T_q, cfg.H_q, dtype=torch.float32, device=dev)

        def pmstep(i, s):
            assert g.gqa_attn_decode_paged_multi(qd, kps[i % nc], vps[i % nc], td, ld, cfg.B, T_q,
                                                 kp.shape[0], page, table.shape[1], cfg.H_q,
                                                 cfg.H_kv, cfg.d, cfg.scale, n, ws, out, lse,
                                                 s) == g.GQA_OK
            assert g.gqa_attn_decode_combine(ws, cfg.B * T_q, cfg.H_q, cfg.d, n, out, lse,
                                             s) == g.GQA_OK

        for c in range(nc):
            pmstep(c, stream)
        ms, rep = timed(pmstep, nc)
        gbs = kv_bytes / (ms * 1e-3) / 1e9
        return {"metric": f"paged multi-token decode KV GB/s ({cfg.name}, page {page}, T_q={T_q})",
                "value": round(gbs, 2), "unit": "GB/s", "ms_per_step": round(ms, 5),
                "repeats": rep, "steps": steps, "n_split": n, "kv_bytes": kv_bytes,
                "frac_of_" + peak_kind + "_hbm": round(gbs / hbm_gbs, 4),
                "l2": f"{nc} rotating page pools", "dtype": "bf16", "data": "synthetic"}

    if name.startswith("decode_paged"):
        cfg = inputs.LLAMA70B_DECODE
        page = int(name[len("decode_paged"):])
        q, k, v, lens = inputs.decode_inputs_for(cfg, seed=0)
        kv_bytes = 2 * int(lens.sum()) * cfg.H_kv * cfg.d * 2
        kp, vp, table = _shuffled_pages(k, v, page, seed=0)
        qd, ld, td = q.to(dev), lens.to(dev), table.to(dev)
        nc = n_copies(kv_bytes)
        kps = [kp.to(dev) for _ in range(nc)]
        vps = [vp.to(dev) for _ in range(nc)]
        n = g.paged_default_splits(cfg.B, cfg.H_kv, cfg.S_max, cfg.d, page)
        ws = g.decode_workspace(cfg.B, cfg.H_q, cfg.d, n, dev)
        out = torch.empty(cfg.B, cfg.H_q, cfg.d, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(cfg.B, cfg.H_q, dtype=torch.float32, device=dev)

        def pstep(i, s):
            assert g.gqa_attn_decode_paged(qd, kps[i % nc], vps[i % nc], td, ld, cfg.B, kp.shape[0],
                                           page, table.shape[1], cfg.H_q, cfg.H_kv, cfg.d,
                                           cfg.scale, n, ws, out, lse, s) == g.GQA_OK
            assert g.gqa_attn_decode_combine(ws, cfg.B, cfg.H_q, cfg.d, n, out, lse,
                                             s) == g.GQA_OK

        for c in range(nc):
            pstep(c, stream)
        ms, rep = timed(pstep, nc)
        gbs = kv_bytes / (ms * 1e-3) / 1e9
        return {"metric": f"paged decode KV GB/s ({cfg.name}, page {page}, shuffled pages)",
                "value": round(gbs, 2), "unit": "GB/s", "ms_per_step": round(ms, 5),
                "repeats": rep, "steps": steps, "n_split": n, "kv_bytes": kv_bytes,
                "frac_of_" + peak_kind + "_hbm": round(gbs / hbm_gbs, 4),
                "l2": f"{nc} rotating page pools", "dtype": "bf16", "data": "synthetic"}

    # prefill workloads
    if name == "prefill_64k":
        cfg = inputs.PREFILL_64K
        q, k, v = inputs.prefill_inputs_for(cfg, seed=0)
        B, T_q, S_kv, H_q, H_kv, d, W, L = cfg.B, cfg.S, cfg.S, cfg.H_q, cfg.H_kv, cfg.d, -1, cfg.S
        label = cfg.name
    elif name in ("prefill_d64", "prefill_d32"):
        # the Llama3-70B-shaped 8K causal prefill at a smaller head dimension
        d = 64 if name == "prefill_d64" else 32
        B, T_q, S_kv, H_q, H_kv, W, L = 1, 8192, 8192, 64, 8, -1, 8192
        q, k, v = inputs.prefill_inputs(B, T_q, H_q, H_kv, d, seed=0)
        label = f"prefill_causal_s8192_hq64_hkv8_d{d}"
    elif name == "prefill_window":
        cfg = inputs.LLAMA70B_PREFILL_8K
        q, k, v = inputs.prefill_inputs_for(cfg, seed=0)
        B, T_q, S_kv, H_q, H_kv, d, W, L = cfg.B, cfg.S, cfg.S, cfg.H_q, cfg.H_kv, cfg.d, 4096, cfg.S
        label = "prefill_causal_llama70b_s8192_window4096"
    else:  # chunk of 2048 queries ending a 32768-token sequence
        B, T_q, S_kv, H_q, H_kv, d, W, L = 1, 2048, 32768, 64, 8, 128, -1, 32768
        gen = torch.Generator().manual_seed(0)
        q = torch.randn(B, T_q, H_q, d, generator=gen).to(torch.bfloat16)
        k = torch.randn(B, S_kv, H_kv, d, generator=gen).to(torch.bfloat16)
        v = torch.randn(B, S_kv, H_kv, d, generator=gen).to(torch.bfloat16)
        label = "prefill_chunk_llama70b_t2048_at_32768"
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty_like(qd)
    lse = torch.empty(B, H_q, T_q, dtype=torch.float32, device=dev)
    lens = torch.full((B,), L, dtype=torch.int32, device=dev)
    # visible (query, key) pairs: row a = L - T_q + i sees keys max(0, a - W) .. a
    a = torch.arange(L - T_q, L, dtype=torch.float64)
    vis = (a + 1) if W < 0 else torch.minimum(a, torch.full_like(a, W)) + 1
    flops = 4.0 * d * H_q * B * float(vis.sum())

    causal_only = name in ("prefill_64k", "prefill_d64", "prefill_d32")
    n_part = 1 if causal_only else g.gqa_attn_prefill_chunk_default_parts(B, T_q, S_kv, H_q, H_kv)
    ws = torch.empty(max(1, g.gqa_attn_prefill_chunk_workspace_bytes(B, T_q, H_q, d, n_part)),
                     dtype=torch.uint8, device=dev)

    def step(i, s):
        if causal_only:
            st = g.gqa_attn_prefill_causal(qd, kd, vd, B, T_q, H_q, H_kv, d, scale, out, lse, s)
        else:
            st = g.gqa_attn_prefill_chunk_split(qd, kd, vd, lens, B, T_q, S_kv, H_q, H_kv, d, scale,
                                                W, n_part, ws, out, lse, s)
        assert st == g.GQA_OK

    ms, rep = timed(step)
    tf = flops / (ms * 1e-3) / 1e12
    return {"metric": f"prefill TFLOPS ({label})", "value": round(tf, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "repeats": rep, "steps": steps, "flops_per_step": flops,
            "n_part": n_part,
            "frac_of_" + peak_kind + "_bf16": round(tf / bf16_tf, 4), "dtype": "bf16",
            "data": "synthetic"}


def emit(line, args, name):
    """Print the JSON line; with --results-dir also write it to
    <dir>/<name>_<UTC time>.json."""
    text = json.dumps(line)
    print(text, flush=True)
    if args.results_dir:
        os.makedirs(args.results_dir, exist_ok=True)
        stamp = time.strftime("%Y%m%dT%H%M%SZ", time.gmtime())
        with open(os.path.join(args.results_dir, f"{name}_{stamp}.json"), "w") as f:
            f.write(text + "\n")


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="time the headline step only, without the other workloads under "
                         "'configs' (for profiler captures); the JSON line is partial")
    ap.add_argument("--workload", choices=WORKLOADS, default=None,
                    help="measure one further workload instead of the headline step")
    ap.add_argument("--only", choices=["decode", "prefill"], default=None,
                    help="run one leg of the headline step only (for profiler captures); "
                         "the JSON line is partial")
    ap.add_argument("--seed", type=int, default=0,
                    help="seed of the synthetic inputs of the headline step, its configs and "
                         "the reference arm (the oracle parity uses the same inputs)")
    ap.add_argument("--splits", type=int, default=None,
                    help="split count of the headline decode (default: "
                         "gqa_attn_decode_default_splits)")
    ap.add_argument("--results-dir", default=None,
                    help="also write the JSON line to a file in this directory")
    args = ap.parse_args()
    if args.splits is not None and args.splits < 1:
        ap.error("--splits must be >= 1")
    if args.warmup < 3:
        args.warmup = 3
    args.steps = max(1, args.steps)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.workload is not None:
        if rank == 0:
            emit(run_workload(args.workload, args), args, args.workload)
        return 0
    if args.impl == "reference":
        if world > 1 and rank != 0:
            return 0
        emit(run_reference(args, rank, world), args, "reference")
        return 0
    if world > 1:
        import torch
        import torch.distributed as tdist

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
        dist = tdist
    try:
        line = run_ours(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()
    if rank == 0 and line is not None:
        emit(line, args, "step" if args.only is None else args.only)
    return 0


if __name__ == "__main__":
    sys.exit(main())
