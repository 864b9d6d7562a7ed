#!/usr/bin/env python3
"""Benchmark of the grouped-query attention forward hot path on one GB300.

One step = one pass of the whole path on seeded synthetic inputs:
  * decode  : Llama3-70B-shaped GQA decode, B=1, H_q=64, H_kv=8, d=128,
              ctx 32768 -- split-KV kernel + log-sum-exp combine;
  * prefill : Llama3-70B-shaped causal GQA prefill, B=1, S=8192, H_q=64,
              H_kv=8, d=128.
``value`` is the decode leg's KV-cache throughput (GB/s of K and V bytes read,
inputs resident in HBM; rotating K/V copies, at least 1.5 GiB of them, so
that no step finds its inputs in L2); the prefill leg's TFLOP/s (causal FLOPs only) is reported beside
it under ``prefill``.

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
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode KV GB/s (% HBM peak); causal prefill TFLOPS (% bf16 peak)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


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


# ------------------------------------------------------------------- ours ---
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


def _time_region(torch, fn, steps, stream):
    """Events around `steps` back-to-back calls fn(i); returns mean ms per call."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        fn(i)
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / steps


# Decode inputs rotate through copies of the cache so that a copy is read again
# only after at least ROTATION_BYTES of other cache reads (12 x the 126 MB L2).
# The decode sweep loads K/V evict-first in L2, which leaves the lines that a
# step prefetched at normal priority; with 3 copies (384 MiB) some of them were
# still in L2 when their copy came round again (measured 1.1 us faster per
# step than with 12 copies), so a shorter rotation would overstate the rate.
ROTATION_BYTES = 3 << 29


def n_copies(bytes_per_copy):
    return max(2, -(-ROTATION_BYTES // bytes_per_copy))


def run_ours(args, rank, world, dist):
    import torch

    import gqa_attention_gb300 as g
    from gqa_attention_gb300 import inputs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    g.load()
    stream = torch.cuda.current_stream()
    hbm_gbs, bf16_tf, bf16_tf_sus, peak_kind = _peaks()

    # ---------------- decode leg (Llama3-70B decode, ctx 32768) ----------------
    dc = inputs.LLAMA70B_DECODE
    q, k, v, lens = inputs.decode_inputs_for(dc, seed=0)
    kv_bytes = 2 * int(lens.sum()) * dc.H_kv * dc.d * 2
    qd, ld = q.to(dev), lens.to(dev)
    N_KV_COPIES = n_copies(kv_bytes)
    kds = [k.to(dev) for _ in range(N_KV_COPIES)]
    vds = [v.to(dev) for _ in range(N_KV_COPIES)]
    n_split = g.gqa_attn_decode_default_splits(dc.B, dc.H_kv, dc.S_max, dc.d)
    ws = g.decode_workspace(dc.B, dc.H_q, dc.d, n_split, dev)
    out = torch.empty(dc.B, dc.H_q, dc.d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(dc.B, dc.H_q, dtype=torch.float32, device=dev)

    def split_only(i):
        st = g.gqa_attn_decode(qd, kds[i % N_KV_COPIES], vds[i % N_KV_COPIES], ld, dc.B,
                               dc.S_max, dc.H_q, dc.H_kv, dc.d, dc.scale, n_split, ws, out, lse,
                               stream)
        if st:
            raise RuntimeError(f"decode failed: {g.status_str(st)}")

    def decode_step(i):
        # split kernel + combine kernel back to back (the combine may overlap the
        # split kernel's tail through programmatic dependent launch)
        split_only(i)
        st = g.gqa_attn_decode_combine(ws, dc.B, dc.H_q, dc.d, n_split, out, lse, stream)
        if st:
            raise RuntimeError(f"combine failed: {g.status_str(st)}")

    # ---------------- prefill leg (Llama3-70B causal prefill, S 8192) ----------
    pc = inputs.LLAMA70B_PREFILL_8K
    pq, pk, pv = inputs.prefill_inputs_for(pc, seed=0)
    pqd, pkd, pvd = (x.to(dev) for x in (pq, pk, pv))
    pout = torch.empty_like(pqd)
    plse = torch.empty(pc.B, pc.H_q, pc.S, dtype=torch.float32, device=dev)
    causal_flops = 4.0 * pc.d * pc.H_q * pc.B * pc.S * (pc.S + 1) / 2
    prefill_ok = g.gqa_attn_prefill_causal(pqd, pkd, pvd, pc.B, pc.S, pc.H_q, pc.H_kv, pc.d,
                                           pc.scale, pout, plse, stream) == g.GQA_OK
    torch.cuda.synchronize()

    def prefill_step(i):
        st = g.gqa_attn_prefill_causal(pqd, pkd, pvd, pc.B, pc.S, pc.H_q, pc.H_kv, pc.d,
                                       pc.scale, pout, plse, stream)
        if st:
            raise RuntimeError(f"prefill failed: {g.status_str(st)}")

    run_decode = args.only in (None, "decode")
    if args.only == "decode":
        prefill_ok = False

    # ---------------- warm-up ----------------
    for i in range(args.warmup):
        if run_decode:
            decode_step(i)
            split_only(i)
        if prefill_ok:
            prefill_step(i)
    torch.cuda.synchronize()
    if g.gqa_last_device_error(stream) != g.GQA_OK:
        raise RuntimeError("device error during warm-up")

    # ---------------- timed region ----------------
    with ClockSampler(dev.index) as clk:
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        dec_ms = _time_region(torch, decode_step, args.steps, stream) if run_decode else float("nan")
        split_ms = _time_region(torch, split_only, args.steps, stream) if run_decode else float("nan")
        pre_ms = _time_region(torch, prefill_step, args.steps, stream) if prefill_ok else None
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        wall_s = time.perf_counter() - t_wall
    clocks = clk.summary()
    if g.gqa_last_device_error(stream) != g.GQA_OK:
        raise RuntimeError("device error during the timed region")

    # ---------------- end to end through the C ABI from pinned host buffers -----
    hq, hk, hv, hl = (x.pin_memory() for x in (q, k, v, lens))
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hl))
    d2h = hout.numel() * hout.element_size() + hlse.numel() * hlse.element_size()

    def e2e_step(i):
        qd.copy_(hq, non_blocking=True)
        kds[0].copy_(hk, non_blocking=True)
        vds[0].copy_(hv, non_blocking=True)
        ld.copy_(hl, non_blocking=True)
        decode_step(0)
        hout.copy_(out, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 50))
    if run_decode:
        _time_region(torch, e2e_step, 2, stream)
        e2e_ms = _time_region(torch, e2e_step, e2e_steps, stream)
    else:
        e2e_ms = float("nan")

    # max over ranks
    dec_ms, split_ms, pre_ms_max, e2e_ms = max_over_ranks(
        [dec_ms, split_ms, pre_ms or 0.0, e2e_ms], dist, dev)
    pre_ms = pre_ms_max if pre_ms is not None else None
    if rank != 0:
        return None

    value = whole_job_rate(world, kv_bytes, dec_ms * 1e-3) / 1e9
    ws_bytes = g.gqa_attn_decode_workspace_bytes(dc.B, dc.H_q, dc.d, n_split) if n_split > 1 else 0
    all_bytes = (kv_bytes + dc.B * dc.H_q * dc.d * 2          # K/V read, Q read
                 + 2 * ws_bytes                                # partials written, read back
                 + dc.B * dc.H_q * (dc.d * 2 + 4))             # O (bf16) and LSE written
    achieved = kv_bytes / (split_ms * 1e-3) / 1e9
    traffic = _recorded_traffic("decode_split_llama70b_ctx32768.md",
                                ["decode.cu", "common.cuh", "internal.h"])
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dec_ms + (pre_ms or 0.0), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded torch.randn, rounded to bf16)",
        "config": {
            "workload": f"{dc.name} (value) + {pc.name} (prefill)",
            "decode": {"B": dc.B, "H_q": dc.H_q, "H_kv": dc.H_kv, "d": dc.d, "ctx": dc.S_max,
                       "n_split": n_split, "kv_bytes": kv_bytes,
                       # every byte the two launches move: K/V, Q, the split partials
                       # written and read back, O and LSE
                       "all_bytes": all_bytes,
                       "all_bytes_GBs": round(all_bytes / (dec_ms * 1e-3) / 1e9, 2),
                       "ms_split_plus_combine": round(dec_ms, 5),
                       "ms_split_kernel": round(split_ms, 5),
                       "hbm_frac_of_" + peak_kind: round(value / world / hbm_gbs, 4),
                       "hbm_frac_of_nominal_8TBs": round(value / world / 8000.0, 4)},
            "prefill": {"B": pc.B, "S": pc.S, "H_q": pc.H_q, "H_kv": pc.H_kv, "d": pc.d},
            "l2": (f"decode: {N_KV_COPIES} rotating K/V copies ({N_KV_COPIES * kv_bytes >> 20} MiB), "
                   "a copy is read again only after >= 1.5 GiB (12 x L2) of other cache reads; "
                   "prefill inputs (160 MiB) exceed L2"),
            "timing": "CUDA events around K back-to-back steps on the launching stream",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "clocks": clocks,
        "roofline": {
            "kernel": "gqa_decode_split_kernel",
            "bound": "hbm",
            "achieved": round(achieved, 2),
            "peak": hbm_gbs,
            "unit": "GB/s",
            "frac": round(achieved / hbm_gbs, 4),
            "peak_kind": peak_kind,
            "traffic": traffic,
            "algorithmic_bytes_per_launch": kv_bytes,
        },
        "gpu_launches": args.steps * (3 + (1 if prefill_ok else 0)),
        "e2e": {"value": round(whole_job_rate(world, kv_bytes, e2e_ms * 1e-3) / 1e9, 2),
                "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4)},
        "wall_s_timed_region": round(wall_s, 3),
    }
    if pre_ms is not None:
        tflops = causal_flops / (pre_ms * 1e-3) / 1e12
        line["prefill"] = {
            "value": round(whole_job_rate(world, causal_flops, pre_ms * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "ms": round(pre_ms, 4),
            "causal_flops": causal_flops,
            "roofline": {"kernel": "gqa_prefill_causal_kernel", "bound": "tensor",
                         "achieved": round(tflops, 2), "peak": bf16_tf, "unit": "TFLOP/s",
                         "frac": round(tflops / bf16_tf, 4),
                         "peak_kind": peak_kind + " (burst)",
                         "frac_of_sustained": round(tflops / bf16_tf_sus, 4),
                         "traffic": _recorded_traffic("prefill_causal_llama70b_s8192.md",
                                                      ["prefill.cu", "tcgen05.cuh", "common.cuh",
                                                       "internal.h"])},
        }
    else:
        line["prefill"] = None
    # the oracle on the host cores: a single-GPU figure, taken on rank 0 at N = 1
    line["cpu_baseline"] = (cpu_baseline(args, steps=5)
                            if not args.no_cpu_baseline and world == 1 else None)
    return line


# ---------------------------------------------------- further workloads ---
WORKLOADS = ("decode_tiny", "decode_ragged", "decode_paged16", "decode_paged128", "decode_fp8",
             "decode_fp8_ragged", "decode_multi2", "decode_multi4", "decode_multi8", "decode_multi16",
             "decode_paged16_multi8", "decode_paged128_multi8", "prefill_64k", "prefill_window",
             "prefill_chunk")


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


def run_workload(name, args):
    """One JSON line for a workload other than the headline step (same timing rules)."""
    import torch

    import gqa_attention_gb300 as g
    from gqa_attention_gb300 import inputs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    g.load()
    stream = torch.cuda.current_stream()
    hbm_gbs, bf16_tf, _, peak_kind = _peaks()
    steps = max(1, args.steps)

    def timed(fn):
        for i in range(max(3, args.warmup)):
            fn(i)
        torch.cuda.synchronize()
        ms = _time_region(torch, fn, steps, stream)
        if g.gqa_last_device_error(stream) != g.GQA_OK:
            raise RuntimeError("device error")
        return ms

    if name.startswith("decode_fp8"):
        cfg = inputs.LLAMA70B_DECODE if name == "decode_fp8" else inputs.LLAMA70B_DECODE_RAGGED
        q, k8, v8, ks, vs, lens = inputs.decode_inputs_fp8(cfg.B, cfg.H_q, cfg.H_kv, cfg.d,
                                                           cfg.S_max, seed=0, ragged=cfg.ragged)
        # bytes the sweep must read: E4M3 codes + one fp32 scale per token, for K and V
        kv_bytes = 2 * int(lens.sum()) * (cfg.H_kv * cfg.d + 4)
        copies = n_copies(kv_bytes)
        qd, ld = q.to(dev), lens.to(dev)
        caches = [tuple(x.to(dev) for x in (k8, v8, ks, vs)) for _ in range(copies)]
        n = 3 * g.gqa_attn_decode_default_splits(cfg.B, cfg.H_kv, cfg.S_max, cfg.d)
        ws = g.decode_workspace(cfg.B, cfg.H_q, cfg.d, n, dev)
        out = torch.empty(cfg.B, cfg.H_q, cfg.d, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(cfg.B, cfg.H_q, dtype=torch.float32, device=dev)

        def fstep(i):
            kc, vc, ksc, vsc = caches[i % copies]
            assert g.gqa_attn_decode_fp8(qd, kc, vc, ksc, vsc, ld, cfg.B, cfg.S_max, cfg.H_q,
                                         cfg.H_kv, cfg.d, cfg.scale, n, ws, out, lse,
                                         stream) == g.GQA_OK
            assert g.gqa_attn_decode_combine(ws, cfg.B, cfg.H_q, cfg.d, n, out, lse,
                                             stream) == g.GQA_OK

        ms = timed(fstep)
        gbs = kv_bytes / (ms * 1e-3) / 1e9
        bf16_equiv = 2 * int(lens.sum()) * cfg.H_kv * cfg.d * 2
        return {"metric": f"FP8-cache decode GB/s ({cfg.name})", "value": round(gbs, 2),
                "unit": "GB/s", "ms_per_step": round(ms, 5), "steps": steps, "n_split": n,
                "fp8_bytes": kv_bytes, "bf16_equivalent_GBs": round(bf16_equiv / (ms * 1e-3) / 1e9, 2),
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

        def mstep(i):
            assert g.gqa_attn_decode_multi(qd, kds[i % nc], vds[i % nc], ld, cfg.B, T_q, cfg.S_max,
                                           cfg.H_q, cfg.H_kv, cfg.d, cfg.scale, n, ws, out, lse,
                                           stream) == g.GQA_OK
            assert g.gqa_attn_decode_combine(ws, cfg.B * T_q, cfg.H_q, cfg.d, n, out, lse,
                                             stream) == g.GQA_OK

        def cstep(i):
            assert g.gqa_attn_prefill_chunk(qd, kds[i % nc], vds[i % nc], ld, cfg.B, T_q, cfg.S_max,
                                            cfg.H_q, cfg.H_kv, cfg.d, cfg.scale, -1, out, lse_c,
                                            stream) == g.GQA_OK

        ms = timed(mstep)
        ms_chunk = timed(cstep)
        gbs = kv_bytes / (ms * 1e-3) / 1e9
        return {"metric": f"multi-token decode KV GB/s ({cfg.name}, T_q={T_q})",
                "value": round(gbs, 2),
                "unit": "GB/s", "ms_per_step": round(ms, 5), "steps": steps, "n_split": n,
                "kv_bytes": kv_bytes, "frac_of_" + peak_kind + "_hbm": round(gbs / hbm_gbs, 4),
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

        def pmstep(i):
            assert g.gqa_attn_decode_paged_multi(qd, kps[i % nc], vps[i % nc], td, ld, cfg.B, T_q,
                                                 kp.shape[0], page, table.shape[1], cfg.H_q,
                                                 cfg.H_kv, cfg.d, cfg.scale, n, ws, out, lse,
                                                 stream) == g.GQA_OK
            assert g.gqa_attn_decode_combine(ws, cfg.B * T_q, cfg.H_q, cfg.d, n, out, lse,
                                             stream) == g.GQA_OK

        ms = timed(pmstep)
        gbs = kv_bytes / (ms * 1e-3) / 1e9
        return {"metric": f"paged multi-token decode KV GB/s ({cfg.name}, page {page}, T_q={T_q})",
                "value": round(gbs, 2), "unit": "GB/s", "ms_per_step": round(ms, 5),
                "steps": steps, "n_split": n, "kv_bytes": kv_bytes,
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

        def pstep(i):
            assert g.gqa_attn_decode_paged(qd, kps[i % nc], vps[i % nc], td, ld, cfg.B, kp.shape[0],
                                           page, table.shape[1], cfg.H_q, cfg.H_kv, cfg.d,
                                           cfg.scale, n, ws, out, lse, stream) == g.GQA_OK
            assert g.gqa_attn_decode_combine(ws, cfg.B, cfg.H_q, cfg.d, n, out, lse,
                                             stream) == g.GQA_OK

        ms = timed(pstep)
        gbs = kv_bytes / (ms * 1e-3) / 1e9
        return {"metric": f"paged decode KV GB/s ({cfg.name}, page {page}, shuffled pages)",
                "value": round(gbs, 2), "unit": "GB/s", "ms_per_step": round(ms, 5),
                "steps": steps, "n_split": n, "kv_bytes": kv_bytes,
                "frac_of_" + peak_kind + "_hbm": round(gbs / hbm_gbs, 4),
                "l2": f"{nc} rotating page pools", "dtype": "bf16", "data": "synthetic"}

    if name.startswith("decode"):
        cfg = inputs.TINY_DECODE if name == "decode_tiny" else inputs.LLAMA70B_DECODE_RAGGED
        q, k, v, lens = inputs.decode_inputs_for(cfg, seed=0)
        kv_bytes = 2 * int(lens.sum()) * cfg.H_kv * cfg.d * 2
        copies = n_copies(kv_bytes)
        qd, ld = q.to(dev), lens.to(dev)
        kds = [k.to(dev) for _ in range(copies)]
        vds = [v.to(dev) for _ in range(copies)]
        n = g.gqa_attn_decode_default_splits(cfg.B, cfg.H_kv, cfg.S_max, cfg.d)
        ws = g.decode_workspace(cfg.B, cfg.H_q, cfg.d, n, dev)
        out = torch.empty(cfg.B, cfg.H_q, cfg.d, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(cfg.B, cfg.H_q, dtype=torch.float32, device=dev)

        def step(i):
            c = i % copies
            assert g.gqa_attn_decode(qd, kds[c], vds[c], ld, cfg.B, cfg.S_max, cfg.H_q, cfg.H_kv,
                                     cfg.d, cfg.scale, n, ws, out, lse, stream) == g.GQA_OK
            if n > 1:
                assert g.gqa_attn_decode_combine(ws, cfg.B, cfg.H_q, cfg.d, n, out, lse,
                                                 stream) == g.GQA_OK

        ms = timed(step)
        gbs = kv_bytes / (ms * 1e-3) / 1e9
        return {"metric": f"decode KV GB/s ({cfg.name})", "value": round(gbs, 2), "unit": "GB/s",
                "ms_per_step": round(ms, 5), "steps": steps, "n_split": n, "kv_bytes": kv_bytes,
                "frac_of_" + peak_kind + "_hbm": round(gbs / hbm_gbs, 4),
                "l2": f"{copies} rotating K/V copies",
                "dtype": "bf16", "data": "synthetic"}

    # prefill workloads
    if name == "prefill_64k":
        cfg = inputs.PREFILL_64K
        q, k, v = inputs.prefill_inputs_for(cfg, seed=0)
        B, T_q, S_kv, H_q, H_kv, d, W, L = cfg.B, cfg.S, cfg.S, cfg.H_q, cfg.H_kv, cfg.d, -1, cfg.S
        label = cfg.name
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

    n_part = 1 if name == "prefill_64k" else g.gqa_attn_prefill_chunk_default_parts(
        B, T_q, S_kv, H_q, H_kv)
    ws = torch.empty(max(1, g.gqa_attn_prefill_chunk_workspace_bytes(B, T_q, H_q, d, n_part)),
                     dtype=torch.uint8, device=dev)

    def step(i):
        if name == "prefill_64k":
            st = g.gqa_attn_prefill_causal(qd, kd, vd, B, T_q, H_q, H_kv, d, scale, out, lse, stream)
        else:
            st = g.gqa_attn_prefill_chunk_split(qd, kd, vd, lens, B, T_q, S_kv, H_q, H_kv, d, scale,
                                                W, n_part, ws, out, lse, stream)
        assert st == g.GQA_OK

    ms = timed(step)
    tf = flops / (ms * 1e-3) / 1e12
    return {"metric": f"prefill TFLOPS ({label})", "value": round(tf, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "steps": steps, "flops_per_step": flops,
            "n_part": n_part,
            "frac_of_" + peak_kind + "_bf16": round(tf / bf16_tf, 4), "dtype": "bf16",
            "data": "synthetic"}


# ------------------------------------------------------ CPU oracle baseline --
def cpu_baseline(args, steps=1):
    """Time the fp64 oracle on the host cores on a bounded sample of the decode workload."""
    import oracle
    from gqa_attention_gb300 import inputs

    oracle.build()
    dc = inputs.LLAMA70B_DECODE
    q, k, v, lens = inputs.decode_inputs_for(dc, seed=0)
    kv_bytes = 2 * int(lens.sum()) * dc.H_kv * dc.d * 2
    cores = os.cpu_count() or 1
    times = []
    for _ in range(max(1, steps)):
        t0 = time.perf_counter()
        oracle.decode(q, k, v, lens, dc.scale, nthreads=cores)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    # the same sample on one core (the oracle's thread pool of one)
    t0 = time.perf_counter()
    oracle.decode(q, k, v, lens, dc.scale, nthreads=1)
    t1 = time.perf_counter() - t0
    return {"value": round(kv_bytes / t / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"whole {dc.name} decode (all 64 query heads, 32768 keys), fp64, "
                      f"median of {len(times)} run(s), {t:.3f} s each",
            "value_1core": round(kv_bytes / t1 / 1e9, 4)}


def run_reference(args, rank, world):
    """The oracle as the reference arm: K timed steps of the whole decode workload on CPU."""
    if rank != 0:
        return None
    import oracle
    from gqa_attention_gb300 import inputs

    oracle.build()
    dc = inputs.LLAMA70B_DECODE
    q, k, v, lens = inputs.decode_inputs_for(dc, seed=0)
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
                         "kind": "oracle",
                         "sample": f"whole {dc.name} decode per step (fp64 oracle)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=WORKLOADS, default=None,
                    help="measure one further workload instead of the headline step")
    ap.add_argument("--only", choices=["decode", "prefill"], default=None,
                    help="run one leg only (for profiler captures); the JSON line is partial")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.workload is not None:
        if rank == 0:
            print(json.dumps(run_workload(args.workload, args)), flush=True)
        return 0
    if args.impl == "reference":
        if world > 1 and rank != 0:
            return 0
        line = run_reference(args, rank, world)
        print(json.dumps(line), flush=True)
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
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
