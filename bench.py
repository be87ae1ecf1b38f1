#!/usr/bin/env python3
"""Benchmark of one MLA decode step (attend -> merge -> value/gate) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints ONE JSON line (rank 0).  A step is one pass of the whole path over
one batch of the workload (default: 64 single-token requests, 12 heads,
context lengths uniform in [1024, 8192], fp8 KV), inputs resident in HBM.
L2 is flushed (a 256 MB write) before every timed step; only the step is
inside the CUDA events.  ``value`` is query rows (tokens) per second over
all ranks, the step's launches replayed from one captured CUDA graph;
``kernels_us`` and the roofline come from a second, eager pass with an
event around each launch.  ``e2e`` repeats the step through the public API with the step's
inputs copied from pinned host memory and its output read back, inside
the timed region.  ``roofline`` is the attend kernel's algorithmic HBM bytes
per launch over its event-timed duration, against the measured copy
bandwidth.  ``cpu_baseline`` times the plain C fp64 oracle on the host
cores over a bounded sample of the same workload.

Multi-GPU (torchrun): every rank runs an independent replica of the step
(the path has no cross-GPU exchange here); value = all ranks' rows / the
slowest rank's time.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import mla_decode_paged_gb300 as mla  # noqa: E402
from mla_decode_paged_gb300 import workloads as W  # noqa: E402

METRIC = "mla_decode_tokens_per_s"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, device="cpu"):
    """Element-wise max of per-rank floats across the process group (the
    slowest rank's times); identity without one."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def aggregate_value(rows_per_step, steps, world_size, max_seconds):
    """Whole-job throughput: query rows of every rank over the slowest rank's time."""
    return rows_per_step * steps * world_size / max_seconds


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _spec(name):
    for s in W.WORKLOADS:
        if s.name == name:
            return s
    raise SystemExit("unknown workload %s (have %s)" % (name, [s.name for s in W.WORKLOADS]))


def _plan_splits(plan, R):
    """Splits per request (n_r) of a work plan (items {r, k | n_r << 9 | ...}))."""
    p = plan.numpy().astype(np.int64)
    G = int(p[0])
    it = p[G + 2:].reshape(-1, 4)
    n_r = np.ones(R, dtype=np.int64)
    n_r[it[:, 0]] = (it[:, 1] >> 9) & 511
    return n_r


def _plan_stats(inp, ns, st, page_size=1, plan=None, q_bytes=2):
    """Host-side split counts and the attend kernel's algorithmic bytes
    (KV rows, page / block indices, indptr, q, partials, the work plan)."""
    lens = inp.lengths.cpu().numpy().astype(np.int64)
    if plan is None:
        n_r = np.maximum(1, np.minimum(ns, -(-lens // st)))
    else:
        n_r = _plan_splits(plan, len(lens))
    plan_len = 0 if plan is None else plan.numel()
    used = int(n_r[lens > 0].sum())
    rows_per_req = inp.qlen * inp.heads
    total = int(lens.sum())
    R = len(lens)
    index_bytes = 4 * total if page_size == 1 else 4 * int((-(-lens // page_size)).sum()) + 4 * R
    attend_bytes = (total * 576 + index_bytes + (R + 1) * 4 + R * rows_per_req * 576 * q_bytes + 4 * plan_len
                    + used * rows_per_req * (512 * 2 + 4)
                    + int((ns - n_r).sum() + (lens == 0).sum()) * rows_per_req * 4)
    merge_bytes = used * rows_per_req * (512 * 2 + 4) + ns * R * rows_per_req * 4 + R * rows_per_req * (1024 + 4)
    S = R * inp.qlen
    value_bytes = S * inp.heads * 1024 + inp.heads * 128 * 512 * 2 + 2 * S * inp.heads * 128 * 2 + R * 4
    return dict(used_units=used, attend_bytes=attend_bytes, merge_bytes=merge_bytes, value_bytes=value_bytes,
                kv_tokens=total, attend_flops=2 * total * rows_per_req * (576 + 512))


class Clocks:
    """nvidia-smi sampler running while the timed region runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, directory=None):
        self.index = index
        self.proc = None
        self.path = os.path.join(directory or tempfile.gettempdir(), "mla_bench_clocks_rank%d.csv" % index)

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        self.t0 = time.time()

    def mark(self, begin):
        """Wall-clock bounds of the timed region (samples outside are dropped)."""
        if begin:
            self.r0 = time.time()
        else:
            self.r1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        import datetime
        sm, mx, reasons, total = [], [], set(), 0
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        r0, r1 = getattr(self, "r0", 0.0), getattr(self, "r1", 1e30)
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                clk, cmax = float(parts[2]), float(parts[3])
            except ValueError:
                continue
            total += 1
            if not (r0 - 0.05 <= ts <= r1 + 0.05):
                continue
            sm.append(clk)
            mx.append(cmax)
            for n, v in zip(names[1:], parts[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples_in_region": len(sm), "samples": total}


def run_gpu(args):
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mla.build()
    spec = _spec(args.workload)
    inp = W.make_inputs(spec, dev) if args.page_size == 1 else W.make_block_inputs(spec, dev, args.page_size)
    last = inp.extra.get("last_page_len")
    R, qlen, H = spec.requests, spec.qlen, spec.heads
    S = R * qlen
    ns, st = mla.choose_splits(R, qlen, H, lengths=inp.lengths.cpu())
    # Work plan from the host-known lengths (host metadata, like the split
    # rule above): the requests cut so that every CTA gets about the same
    # number of tiles, at most ns splits each; the partials then need only
    # the splits the plan used.
    plan_h = None
    if not args.no_plan:
        plan_h, ns = mla.plan_units(inp.lengths.cpu(), qlen, H, ns)
    plan = None if plan_h is None else plan_h.to(dev)
    # The query: bf16, or (--q-fp8) e4m3 codes of q * 4 read with q_scale 1/4.
    q_in, q_scale = inp.q, 1.0
    if args.q_fp8:
        q_in, q_scale = (inp.q.float() * 4).to(torch.float8_e4m3fn), 0.25
    stats = _plan_stats(inp, ns, st, args.page_size, plan_h, q_in.element_size())
    stream = torch.cuda.current_stream(dev)

    o = torch.empty((ns, S, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((ns, S, H), dtype=torch.float32, device=dev)
    latent = torch.empty((S, H, 512), dtype=torch.bfloat16, device=dev)
    lse_m = torch.empty((S, H), dtype=torch.float32, device=dev)
    out = torch.empty((S, H * 128), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def step(strm, ev=None):
        if ev:
            ev[0].record(strm)
        mla.attend(q_in, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, ns, st, heads=H, qlen=qlen,
                   o=o, lse=lse, causal=args.causal, page_size=args.page_size, last_page_len=last, plan=plan,
                   q_scale=q_scale, stream=strm)
        if ev:
            ev[1].record(strm)
        if args.three_call:
            mla.merge(o, lse, latent=latent, lse_out=lse_m, stream=strm)
            if ev:
                ev[2].record(strm)
            mla.value_gate(latent, inp.w_uv, inp.gate, inp.lengths, qlen, out=out, stream=strm)
        else:
            mla.merge_value_gate(o, lse, inp.w_uv, inp.gate, inp.lengths, qlen, out=out, latent=latent, stream=strm)
            if ev:
                ev[2].record(strm)
        if ev:
            ev[3].record(strm)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step(stream)
    torch.cuda.synchronize(dev)
    flags = mla.device_status()
    if flags:
        raise SystemExit("device status flags after warm-up: %#x" % flags)
    # The whole step as one CUDA graph (its launches replayed without host work).
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(torch.cuda.current_stream(dev))
    for _ in range(args.warmup):
        flush.fill_(1.0)
        graph.replay()
    torch.cuda.synchronize(dev)

    clocks = Clocks(local, args.clocks_dir)
    clocks.start()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.mark(True)
    gev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush.fill_(1.0)
        gev[k][0].record(stream)
        graph.replay()
        gev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark(False)
    if ws > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    t_step = [e[0].elapsed_time(e[1]) * 1e-3 for e in gev]
    total = sum(t_step)
    # Per-launch times (eager launches, an event pair around each).
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush.fill_(1.0)
        step(stream, evs[k])
    torch.cuda.synchronize(dev)
    t_att = [e[0].elapsed_time(e[1]) * 1e-3 for e in evs]
    t_mrg = [e[1].elapsed_time(e[2]) * 1e-3 for e in evs]
    t_val = [e[2].elapsed_time(e[3]) * 1e-3 for e in evs]
    if mla.device_status():
        raise SystemExit("device status flags after the timed steps")

    # ---- end to end through the public API with host buffers: the step's
    # inputs staged in one pinned host buffer and uploaded with one copy
    # (each piece 256-byte aligned, device views made once), the output read
    # back with one copy.
    host_parts = [q_in, inp.gate, inp.pages, inp.indptr, inp.lengths, last, plan_h]
    offs, total_b = [], 0
    for t in host_parts:
        offs.append(total_b)
        if t is not None:
            total_b += (t.numel() * t.element_size() + 255) // 256 * 256
    stage_h = torch.empty(total_b, dtype=torch.uint8).pin_memory()
    stage_d = torch.empty(total_b, dtype=torch.uint8, device=dev)
    views = []
    for t, off in zip(host_parts, offs):
        if t is None:
            views.append(None)
            continue
        nb = t.numel() * t.element_size()
        stage_h[off:off + nb].copy_(t.detach().cpu().contiguous().view(-1).view(torch.uint8))
        views.append(stage_d[off:off + nb].view(t.dtype).view(t.shape))
    q_d, gate_d, pages_d, indptr_d, lens_d, last_d, plan_d = views
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = total_b
    d2h = out_h.numel() * out_h.element_size()

    # The public calls prepared once (validated, arguments marshalled) over
    # these fixed buffers; each step only launches them.
    att = mla.attend(q_d, inp.kv, pages_d, indptr_d, inp.scale, inp.kv_scale, ns, st, heads=H, qlen=qlen,
                     o=o, lse=lse, causal=args.causal, page_size=args.page_size, last_page_len=last_d, plan=plan_d,
                     q_scale=q_scale, prepare=True)
    mv = None if args.three_call else mla.merge_value_gate(o, lse, inp.w_uv, gate_d, lens_d, qlen, out=out,
                                                           latent=latent, prepare=True)

    def e2e_step():
        stage_d.copy_(stage_h, non_blocking=True)
        att(stream)
        if args.three_call:
            mla.merge(o, lse, latent=latent, lse_out=lse_m, stream=stream)
            mla.value_gate(latent, inp.w_uv, gate_d, lens_d, qlen, out=out, stream=stream)
        else:
            mv(stream)
        out_h.copy_(out, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize(dev)
    e_t = []
    for _ in range(args.steps):
        flush.fill_(1.0)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        e_t.append(a.elapsed_time(b) * 1e-3)
    e2e_total = sum(e_t)
    ok = torch.equal(out_h, out.cpu())
    extra = _time_kv_append(inp, S, flush, dev, stream, args.warmup, min(args.steps, 200))

    if ws > 1:
        total, e2e_total = max_over_ranks([total, e2e_total], dev)
    if rank != 0:
        return None

    hbm, peak_kind = _peaks()
    att = statistics.mean(t_att)
    achieved = stats["attend_bytes"] / att / 1e9
    traffic = _ncu_traffic(spec.name)
    rec = {
        "metric": METRIC,
        "value": aggregate_value(S, args.steps, ws, total),
        "unit": UNIT,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3",    # the attend MMAs (f32 accumulation; config.mma has the rest)
        "data": "synthetic",
        "config": {
            "workload": spec.name, "requests": R, "qlen": qlen, "heads": H, "rows": S,
            "kv_tokens": stats["kv_tokens"], "kv_bytes": stats["kv_tokens"] * 576,
            "num_splits": ns, "split_tokens": st if plan is None else None, "work_units": stats["used_units"],
            "work_plan": "round robin" if plan is None else "host balanced plan (requests cut at tile boundaries so every CTA gets about the same tiles)",
            "l2": "flushed before every timed step (256 MB write, outside the events)",
            "parallelism": "replicas" if ws > 1 else "single-gpu",
            "kv": "fp8-e4m3 paged (page size %d%s)" % (args.page_size, ", block tables" if args.page_size > 1 else ""),
            "mask": "causal within a request" if args.causal else "none",
            "query": "fp8 e4m3 codes of q * 4, q_scale 1/4" if args.q_fp8 else "bf16",
            "mma": "e4m3 x e4m3 -> f32 tcgen05 (attend, two-term split), bf16 mma.sync (W_UV)",
            "launches_per_step": "attend, merge+value/gate" if not args.three_call else "attend, merge, value/gate",
            "timing": "value: CUDA-graph replay of the step; kernels_us / roofline: eager launches, one event pair each",
        },
        "kernels_us": ({"attend": att * 1e6, "merge": statistics.mean(t_mrg) * 1e6,
                        "value_gate": statistics.mean(t_val) * 1e6} if args.three_call else
                       {"attend": att * 1e6, "merge_value_gate": statistics.mean(t_mrg) * 1e6}),
        "kv_tokens_per_s": stats["kv_tokens"] * args.steps * ws / total,
        "roofline": {
            "kernel": "attend", "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)"
            if peak_kind == "measured" else "fallback 6.8 TB/s",
            "algorithmic_bytes_per_launch": stats["attend_bytes"], "traffic": traffic,
        },
        "e2e": {"value": aggregate_value(S, args.steps, ws, e2e_total), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "output_matches_device": bool(ok)},
        "gpu_launches": (3 if args.three_call else 2) * args.steps,
        "extra_ops": extra,
        "clocks": clk,
    }
    if ws == 1 and not args.no_cpu_baseline:
        rec["cpu_baseline"] = cpu_baseline(spec, inp)
    return rec


def _time_kv_append(inp, S, flush, dev, stream, warmup, steps):
    """The cache write of new tokens (not part of the timed step): one new
    token per query row (decode), and a 65,536-token batch (bandwidth).
    Runs after everything else (it overwrites cache rows)."""
    res = {}
    pool = inp.kv.shape[0]
    g = torch.Generator(device=dev).manual_seed(77)
    for name, T in (("decode_tokens", S), ("batch_65536", min(65536, pool))):
        kv_c = torch.randn(T, 512, generator=g, device=dev).to(torch.bfloat16)
        k_pe = torch.randn(T, 64, generator=g, device=dev).to(torch.bfloat16)
        slots = torch.randperm(pool, generator=g, device=dev)[:T].to(torch.int64)
        for _ in range(warmup):
            mla.kv_append(inp.kv, kv_c, k_pe, slots, inp.kv_scale, stream=stream)
        ts = []
        for _ in range(steps):
            flush.fill_(1.0)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            mla.kv_append(inp.kv, kv_c, k_pe, slots, inp.kv_scale, stream=stream)
            b.record(stream)
            ts.append((a, b))
        torch.cuda.synchronize(dev)
        t = statistics.mean(a.elapsed_time(b) * 1e-3 for a, b in ts)
        nbytes = T * (512 * 2 + 64 * 2 + 8 + 576)
        res["kv_append_" + name] = {"tokens": T, "us": t * 1e6, "bytes": nbytes, "GB/s": nbytes / t / 1e9}
    if mla.device_status():
        raise SystemExit("device status flags after kv_append")
    return res


def _ncu_traffic(workload):
    """DRAM bytes per attend launch from the committed ncu summary of this
    workload, if its kernel-source hash matches the current sources (else
    null: the counters describe an older kernel)."""
    p = os.path.join(ROOT, "profiles", "attend_tc_%s.md" % workload)
    if not os.path.exists(p) or os.environ.get("MLA_ATTEND_KERNEL") == "mma":
        return None
    vals = {}
    for line in open(p):
        line = line.strip()
        if ":" in line and line.split(":")[0] in ("kernel_sources_sha256_16", "dram_bytes_per_launch"):
            k, v = line.split(":", 1)
            vals[k] = v.strip()
    if vals.get("kernel_sources_sha256_16") != kernel_sources_hash():
        return None
    return int(vals["dram_bytes_per_launch"])


def kernel_sources_hash():
    """First 16 hex digits of the SHA-256 of the attend kernel's sources
    with comments and whitespace removed (the code the counters describe)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in ("attend_tc.cu", "tc.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "mla_decode_paged_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)      # block comments
        src = re.sub(r"//[^\n]*", " ", src)                     # line comments
        h.update("".join(src.split()).encode())
    return h.hexdigest()[:16]


def cpu_baseline(spec, inp, budget_s=10.0):
    """Time the plain C fp64 oracle on the host cores on a bounded sample of
    the workload's requests (the first requests until ~budget_s of work)."""
    import oracle  # test infrastructure: timed here as the CPU baseline only
    lib = oracle.load_c()
    threads = lib.mla_oracle_threads()
    q = inp.q.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    kv = inp.kv.cpu().numpy()
    pages = inp.pages.cpu().numpy()
    indptr = inp.indptr.cpu().numpy()
    w = inp.w_uv.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    g = inp.gate.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    lens = np.diff(indptr)
    R = len(lens)
    # estimate from a one-request probe, then take as many requests as fit the budget
    t0 = time.perf_counter()
    oracle.decode_step_c(q, kv, pages, indptr, inp.scale, inp.kv_scale, spec.heads, spec.qlen, w, g,
                         requests=[0])
    probe = max(time.perf_counter() - t0, 1e-4)
    per_token = probe / max(1, lens[0])
    n = R
    while n > 1 and per_token * lens[:n].sum() / max(1, min(threads, n)) > budget_s:
        n = max(1, n // 2)
    reqs = list(range(n))
    reps, t0 = 0, time.perf_counter()
    while True:   # repeat the sample until about the budget has been spent
        oracle.decode_step_c(q, kv, pages, indptr, inp.scale, inp.kv_scale, spec.heads, spec.qlen, w, g,
                             requests=reqs)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s or dt / reps * (reps + 1) > 2 * budget_s:
            break
    return {"value": n * spec.qlen * reps / dt, "unit": UNIT, "cores": int(threads), "kind": "oracle",
            "sample": "%d of %d requests (%d KV tokens) x %d repetitions, full path in fp64 C, %.2f s" % (
                n, R, int(lens[:n].sum()), reps, dt)}


def run_reference(args):
    ws, rank, local = _dist()
    if rank != 0:
        return None
    spec = _spec(args.workload)
    inp = W.make_inputs(spec, "cpu")
    times = []
    base = None
    for k in range(args.warmup + args.steps):
        res = cpu_baseline(spec, inp, budget_s=args.ref_budget)
        if k >= args.warmup:
            times.append(res)
        base = res
    vals = [r["value"] for r in times]
    v = statistics.mean(vals) if vals else base["value"]
    S = spec.requests * spec.qlen
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": S / v * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": spec.name, "requests": spec.requests, "qlen": spec.qlen, "heads": spec.heads,
                   "rows": S, "note": "each step times the CPU oracle on a bounded sample of the workload"},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": base["cores"], "kind": "oracle",
                         "sample": base["sample"]},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=W.WORKLOADS[1].name)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--three-call", action="store_true",
                    help="time merge and value/gate as two launches instead of the fused one")
    ap.add_argument("--ref-budget", type=float, default=5.0)
    ap.add_argument("--page-size", type=int, default=1,
                    help="KV cache as block tables of this many rows per block (power of two)")
    ap.add_argument("--q-fp8", action="store_true",
                    help="fp8 e4m3 query codes (q * 4) with q_scale 1/4 instead of the bf16 query")
    ap.add_argument("--no-plan", action="store_true",
                    help="round-robin work units under the split rule instead of the host work plan")
    ap.add_argument("--causal", action="store_true",
                    help="causal mask within a request (row tq sees its first L - qlen + tq + 1 tokens)")
    ap.add_argument("--clocks-dir", default=None,
                    help="where the raw nvidia-smi clock samples go (default: the system temp directory)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rec = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if rec is not None:
        print(json.dumps(rec), flush=True)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1 and args.impl != "reference":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
