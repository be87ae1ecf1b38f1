#!/usr/bin/env python3
"""Benchmark of one MLA decode step (attend -> merge -> value/gate) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints ONE JSON line (rank 0).  A step is one pass of the whole path over
one batch of the workload, inputs resident in HBM.  The default workload is
the largest: 256 requests x 8 query rows (2,048 rows), 12 heads, context
lengths log-uniform in [128, 131072] with 8 empty requests, fp8 KV (about
2.7 GB of KV rows per step).  L2 is flushed (a 256 MB write) before every
timed step; only the step is inside the CUDA events.  ``value`` is query rows
(tokens) per second over all ranks, the step's launches replayed from one
captured CUDA graph; ``kernels_us`` and the roofline come from a second,
eager pass with an event around each launch.  ``e2e`` repeats the step
through the public API with the step's inputs copied from pinned host memory
and its output read back, inside the timed region.  ``roofline`` is the
attend kernel's algorithmic HBM bytes per launch over its event-timed
duration, against the measured copy bandwidth.  ``per_workload`` times the
other full-size workloads the same way (graph-replayed step, event-timed
launches, roofline).  ``cpu_baseline`` times the plain C fp64 oracle on the
host cores over a bounded sample of the same workload, and ``parity_check``
compares the timed run's output with the oracle's on that sample.

Multi-GPU (torchrun): every rank runs an independent replica of the step
(the path has no cross-GPU exchange here); value = all ranks' rows / the
slowest rank's time.
"""

from __future__ import annotations

import argparse
import dataclasses
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


def _spec(name, requests=None):
    """The named workload; with ``requests`` a smaller case of it (the same
    shapes and distributions, the first ``requests`` requests drawn), named
    ``<name>:r<requests>`` (its DRAM traffic is not the full workload's)."""
    for s in W.WORKLOADS:
        if s.name == name:
            if requests:
                s = dataclasses.replace(s, name="%s:r%d" % (s.name, requests), requests=requests,
                                        zero_requests=min(s.zero_requests, requests))
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
        """Wall-clock bounds of a timed region (samples outside every region
        are dropped); call mark(True) / mark(False) around each one."""
        if not hasattr(self, "regions"):
            self.regions = []
        if begin:
            self.regions.append([time.time(), 1e30])
        elif self.regions:
            self.regions[-1][1] = time.time()

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
        regions = getattr(self, "regions", None) or [(getattr(self, "r0", 0.0), getattr(self, "r1", 1e30))]
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
            if not any(r0 - 0.05 <= ts <= r1 + 0.05 for r0, r1 in regions):
                continue
            sm.append(clk)
            mx.append(cmax)
            for n, v in zip(names[1:], parts[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples_in_region": len(sm), "samples": total}


HEADLINE = "ragged_r256_q8_h12"
OTHERS = ("decode_r64_h12", "spec_r128_q4_h12", "long_r32_h96p128")
# The speculative-decode workload's description cuts every request into 8 to
# 32 split-KV partials: 32 splits of 512 tokens under the split rule do that
# for its U[4096, 32768] contexts.
STATED_CUT = ("spec_r128_q4_h12", (32, 512))
# ... and the same 8-32 partials per request cut by the balanced host plan.
STATED_PLAN = (8, 32)   # (min_splits, num_splits)


def _parse_splits(text):
    """``"NS:ST"`` -> (num_splits, split_tokens), or None."""
    if not text:
        return None
    ns, st = (int(x) for x in text.split(":"))
    if ns < 1 or st < 1:
        raise SystemExit("--splits wants two positive integers NS:ST")
    return ns, st


def _plan_ranges(plan_h, num_requests):
    """Per request, its splits' token ranges (row group 0) in a host plan
    ([G, offsets[G + 1], items of 4 int32, then each CTA's first item again])."""
    p = plan_h.to(torch.int64).tolist()
    G = p[0]
    n_items = p[1 + G]
    out = [[] for _ in range(num_requests)]
    for i in range(n_items):
        r, w, s0, c = p[2 + G + 4 * i: 2 + G + 4 * i + 4]
        if (w >> 18) & 8191 == 0:
            out[r].append((s0, s0 + c))
    return out


class Step:
    """One workload's device inputs, split plan, buffers and the step's
    launches (attend, then merge + value/gate)."""

    def __init__(self, spec, args, dev, splits=None, plan_splits=None):
        self.spec, self.args, self.dev = spec, args, dev
        splits = splits or _parse_splits(args.splits)
        if plan_splits is None and splits is None and getattr(args, "plan_splits", None):
            plan_splits = _parse_splits(args.plan_splits)
        inp = W.make_inputs(spec, dev) if args.page_size == 1 else W.make_block_inputs(spec, dev, args.page_size)
        self.inp = inp
        self.last = inp.extra.get("last_page_len")
        R, qlen, H = spec.requests, spec.qlen, spec.heads
        self.S = S = R * qlen
        ns, st = mla.choose_splits(R, qlen, H, lengths=inp.lengths.cpu()) if splits is None else splits
        # Work plan from the host-known lengths (host metadata, like the split
        # rule): the requests cut so that every CTA gets about the same number
        # of tiles, at most ns splits each; the partials then need only the
        # splits the plan used.  A given (num_splits, split_tokens) is timed
        # under the split rule itself.
        self.plan_h = None
        if plan_splits is not None:   # (min_splits, num_splits): a plan honouring a stated partial count
            self.plan_h, ns = mla.plan_units(inp.lengths.cpu(), qlen, H, plan_splits[1], min_splits=plan_splits[0])
        elif not args.no_plan and splits is None:
            self.plan_h, ns = mla.plan_units(inp.lengths.cpu(), qlen, H, ns)
        self.plan = None if self.plan_h is None else self.plan_h.to(dev)
        self.ns, self.st = ns, st
        # The query: bf16, or (--q-fp8) e4m3 codes of q * 4 read with q_scale 1/4.
        self.q_in, self.q_scale = inp.q, 1.0
        if args.q_fp8:
            self.q_in, self.q_scale = (inp.q.float() * 4).to(torch.float8_e4m3fn), 0.25
        self.stats = _plan_stats(inp, ns, st, args.page_size, self.plan_h, self.q_in.element_size())
        self.o = torch.empty((ns, S, H, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((ns, S, H), dtype=torch.float32, device=dev)
        self.latent = torch.empty((S, H, 512), dtype=torch.bfloat16, device=dev)
        self.lse_m = torch.empty((S, H), dtype=torch.float32, device=dev)
        self.out = torch.empty((S, H * 128), dtype=torch.bfloat16, device=dev)

    def launch(self, strm, ev=None):
        a, inp = self.args, self.inp
        if ev:
            ev[0].record(strm)
        mla.attend(self.q_in, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, self.ns, self.st,
                   heads=inp.heads, qlen=inp.qlen, o=self.o, lse=self.lse, causal=a.causal, page_size=a.page_size,
                   last_page_len=self.last, plan=self.plan, q_scale=self.q_scale, stream=strm)
        if ev:
            ev[1].record(strm)
        if a.three_call:
            mla.merge(self.o, self.lse, latent=self.latent, lse_out=self.lse_m, stream=strm)
            if ev:
                ev[2].record(strm)
            mla.value_gate(self.latent, inp.w_uv, inp.gate, inp.lengths, inp.qlen, out=self.out, stream=strm)
        else:
            mla.merge_value_gate(self.o, self.lse, inp.w_uv, inp.gate, inp.lengths, inp.qlen, out=self.out,
                                 latent=self.latent, lse_out=self.lse_m, stream=strm)
            if ev:
                ev[2].record(strm)
        if ev:
            ev[3].record(strm)

    def warm_and_capture(self, flush, warmup):
        """Eager warm-up, a status check, then the step captured as one CUDA
        graph (its launches replayed without host work) and warmed."""
        stream = torch.cuda.current_stream(self.dev)
        for _ in range(warmup):
            flush.fill_(1.0)
            self.launch(stream)
        torch.cuda.synchronize(self.dev)
        flags = mla.device_status()
        if flags:
            raise SystemExit("%s: device status flags after warm-up: %#x" % (self.spec.name, flags))
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.launch(torch.cuda.current_stream(self.dev))
        for _ in range(warmup):
            flush.fill_(1.0)
            self.graph.replay()
        torch.cuda.synchronize(self.dev)

    def time_graph(self, flush, steps):
        """Seconds per graph-replayed step (L2 flushed before each, outside the events)."""
        stream = torch.cuda.current_stream(self.dev)
        gev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for k in range(steps):
            flush.fill_(1.0)
            gev[k][0].record(stream)
            self.graph.replay()
            gev[k][1].record(stream)
        torch.cuda.synchronize(self.dev)
        return [e[0].elapsed_time(e[1]) * 1e-3 for e in gev]

    def time_eager(self, flush, steps):
        """Per-launch seconds (eager launches, an event pair around each)."""
        stream = torch.cuda.current_stream(self.dev)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        for k in range(steps):
            flush.fill_(1.0)
            self.launch(stream, evs[k])
        torch.cuda.synchronize(self.dev)
        if mla.device_status():
            raise SystemExit("%s: device status flags after the timed steps" % self.spec.name)
        return ([e[0].elapsed_time(e[1]) * 1e-3 for e in evs], [e[1].elapsed_time(e[2]) * 1e-3 for e in evs],
                [e[2].elapsed_time(e[3]) * 1e-3 for e in evs])

    def kernels_us(self, t_att, t_mrg, t_val):
        if self.args.three_call:
            return {"attend": statistics.mean(t_att) * 1e6, "merge": statistics.mean(t_mrg) * 1e6,
                    "value_gate": statistics.mean(t_val) * 1e6}
        return {"attend": statistics.mean(t_att) * 1e6, "merge_value_gate": statistics.mean(t_mrg) * 1e6}

    def roofline(self, t_att):
        hbm, peak_kind = _peaks()
        att = statistics.mean(t_att)
        achieved = self.stats["attend_bytes"] / att / 1e9
        return {"kernel": "attend", "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm,
                "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "algorithmic_bytes_per_launch": self.stats["attend_bytes"], "traffic": _ncu_traffic(self.spec.name)}


def run_gpu(args):
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mla.build()
    spec = _spec(args.workload, args.requests)
    step = Step(spec, args, dev)
    inp, S, ns, st, plan = step.inp, step.S, step.ns, step.st, step.plan
    R, qlen, H = spec.requests, spec.qlen, spec.heads
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    step.warm_and_capture(flush, args.warmup)

    clocks = Clocks(local, args.clocks_dir)
    clocks.start()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.mark(True)
    t_step = step.time_graph(flush, args.steps)
    clocks.mark(False)
    if ws > 1:
        torch.distributed.barrier()
    total = sum(t_step)
    t_att, t_mrg, t_val = step.time_eager(flush, args.steps)
    # The timed step's outputs, kept for the comparison with the oracle.
    step.graph.replay()
    torch.cuda.synchronize(dev)
    gpu_out = (step.out.cpu(), step.latent.cpu(), step.lse_m.cpu())

    # ---- end to end through the public API with host buffers.  Each step's
    # inputs (query, gate, page table, indptr, lengths, work plan) are staged
    # in one pinned host buffer and uploaded with one copy (each piece
    # 256-byte aligned, device views made once), and its output is read back
    # with one copy.  Two steps are in flight, as in a serving loop: step
    # k+1's upload (one copy stream) overlaps step k's kernels (the compute
    # stream), and step k's read-back runs on a second copy stream; the
    # staging buffers and outputs alternate between two sets, and each reuse
    # waits for the step that last used the set.  The KV cache and W_UV are
    # resident state.  The timed region runs from the first upload to the
    # last read-back (the KV rows of the default workload exceed L2, so no
    # flush is needed between the overlapped steps).
    q_in, last, plan_h = step.q_in, step.last, step.plan_h
    host_parts = [q_in, inp.gate, inp.pages, inp.indptr, inp.lengths, last, plan_h]
    offs, total_b = [], 0
    for t in host_parts:
        offs.append(total_b)
        if t is not None:
            total_b += (t.numel() * t.element_size() + 255) // 256 * 256
    out, o, lse, latent, lse_m = step.out, step.o, step.lse, step.latent, step.lse_m
    sets = []
    for k in range(2):
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
        out_k = out if k == 0 else torch.empty_like(out)
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        # The public calls prepared once (validated, arguments marshalled)
        # over this set's buffers; each step only launches them.
        att = mla.attend(q_d, inp.kv, pages_d, indptr_d, inp.scale, inp.kv_scale, ns, st, heads=H, qlen=qlen,
                         o=o, lse=lse, causal=args.causal, page_size=args.page_size, last_page_len=last_d,
                         plan=plan_d, q_scale=step.q_scale, prepare=True)
        mv = None if args.three_call else mla.merge_value_gate(o, lse, inp.w_uv, gate_d, lens_d, qlen, out=out_k,
                                                               latent=latent, lse_out=lse_m, prepare=True)
        sets.append(dict(stage_h=stage_h, stage_d=stage_d, att=att, mv=mv, gate_d=gate_d, lens_d=lens_d,
                         out=out_k, out_h=out_h))
    h2d = total_b
    d2h = out.numel() * out.element_size()
    up_stream = torch.cuda.Stream(dev)
    down_stream = torch.cuda.Stream(dev)

    def e2e_run(nsteps):
        ev = lambda: torch.cuda.Event()  # noqa: E731
        up, done, rd = [ev() for _ in range(nsteps)], [ev() for _ in range(nsteps)], [ev() for _ in range(nsteps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        t0.record(up_stream)
        for k in range(nsteps):
            sk = sets[k % 2]
            if k >= 2:
                up_stream.wait_event(done[k - 2])      # step k-2's kernels are done with this set's inputs
            with torch.cuda.stream(up_stream):
                sk["stage_d"].copy_(sk["stage_h"], non_blocking=True)
            up[k].record(up_stream)
            stream.wait_event(up[k])
            if k >= 2:
                stream.wait_event(rd[k - 2])           # step k-2's output has been read back
            sk["att"](stream)
            if args.three_call:
                mla.merge(o, lse, latent=latent, lse_out=lse_m, stream=stream)
                mla.value_gate(latent, inp.w_uv, sk["gate_d"], sk["lens_d"], qlen, out=sk["out"], stream=stream)
            else:
                sk["mv"](stream)
            done[k].record(stream)
            down_stream.wait_event(done[k])
            with torch.cuda.stream(down_stream):
                sk["out_h"].copy_(sk["out"], non_blocking=True)
            rd[k].record(down_stream)
        t1.record(down_stream)
        t1.synchronize()
        return t0.elapsed_time(t1) * 1e-3

    e2e_run(max(2, args.warmup))
    e2e_total = e2e_run(args.steps)
    torch.cuda.synchronize(dev)
    ok = all(torch.equal(sk["out_h"], gpu_out[0]) for sk in sets)

    # ---- the other full-size workloads, each timed the same way (rank 0 of
    # a single-GPU run only: the scaling runs need the headline alone)
    per_workload = {}
    if ws == 1 and not args.no_per_workload and args.workload == HEADLINE and args.requests is None:
        for name in OTHERS:
            other = Step(_spec(name), args, dev)
            other.warm_and_capture(flush, args.warmup)
            clocks.mark(True)
            ts = other.time_graph(flush, args.steps)
            clocks.mark(False)
            oa, om, ov = other.time_eager(flush, args.steps)
            rl = other.roofline(oa)
            per_workload[name] = {
                "requests": other.spec.requests, "qlen": other.spec.qlen, "heads": other.spec.heads,
                "rows": other.S, "kv_tokens": other.stats["kv_tokens"], "num_splits": other.ns,
                "ms_per_step": sum(ts) / len(ts) * 1e3, "tokens_per_s": other.S * len(ts) / sum(ts),
                "kernels_us": other.kernels_us(oa, om, ov),
                "roofline": {k: rl[k] for k in ("achieved", "peak", "unit", "frac", "algorithmic_bytes_per_launch",
                                                "traffic")},
            }
            if name == STATED_CUT[0]:
                # the same workload cut the way its description states (every
                # request into 8-32 partials, split rule), timed the same way
                del other
                torch.cuda.empty_cache()
                other = Step(_spec(name), args, dev, splits=STATED_CUT[1])
                other.warm_and_capture(flush, args.warmup)
                clocks.mark(True)
                ts = other.time_graph(flush, args.steps)
                clocks.mark(False)
                oa, om, ov = other.time_eager(flush, args.steps)
                rl = other.roofline(oa)
                lens = other.inp.lengths.cpu().long()
                n_r = torch.clamp((lens + other.st - 1) // other.st, 1, other.ns)
                per_workload[name]["stated_cut"] = {
                    "num_splits": other.ns, "split_tokens": other.st, "work_plan": "none (split rule)",
                    "partials_per_request": [int(n_r.min()), int(n_r.max())],
                    "ms_per_step": sum(ts) / len(ts) * 1e3, "tokens_per_s": other.S * len(ts) / sum(ts),
                    "kernels_us": other.kernels_us(oa, om, ov),
                    "roofline": {k: rl[k] for k in ("achieved", "frac", "algorithmic_bytes_per_launch")},
                }
                # the same partial count from the balanced plan (at least 8 splits a request)
                del other
                torch.cuda.empty_cache()
                other = Step(_spec(name), args, dev, plan_splits=STATED_PLAN)
                other.warm_and_capture(flush, args.warmup)
                clocks.mark(True)
                ts = other.time_graph(flush, args.steps)
                clocks.mark(False)
                oa, om, ov = other.time_eager(flush, args.steps)
                rl = other.roofline(oa)
                n_r = [len(c) for c in _plan_ranges(other.plan_h, other.spec.requests)]
                per_workload[name]["stated_cut_planned"] = {
                    "num_splits": other.ns, "work_plan": "host plan, at least %d splits a request" % STATED_PLAN[0],
                    "partials_per_request": [min(n_r), max(n_r)],
                    "ms_per_step": sum(ts) / len(ts) * 1e3, "tokens_per_s": other.S * len(ts) / sum(ts),
                    "kernels_us": other.kernels_us(oa, om, ov),
                    "roofline": {k: rl[k] for k in ("achieved", "frac", "algorithmic_bytes_per_launch")},
                }
            del other
            torch.cuda.empty_cache()
    clk = clocks.stop()
    extra = _time_kv_append(S, step.inp.kv_scale, flush, dev, stream, args.warmup, min(args.steps, 200))

    if ws > 1:
        total, e2e_total = max_over_ranks([total, e2e_total], dev)
    if rank != 0:
        return None

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
            "kv_tokens": step.stats["kv_tokens"], "kv_bytes": step.stats["kv_tokens"] * 576,
            "num_splits": ns, "split_tokens": st if plan is None else None, "work_units": step.stats["used_units"],
            "work_plan": "round robin" if plan is None else "host balanced plan (requests cut at tile boundaries so every CTA gets about the same tiles)",
            "l2": "flushed before every timed step (256 MB write, outside the events)",
            "parallelism": "replicas" if ws > 1 else "single-gpu",
            "kv": "fp8-e4m3 paged (page size %d%s)" % (args.page_size, ", block tables" if args.page_size > 1 else ""),
            "mask": "causal within a request" if args.causal else "none",
            "query": "fp8 e4m3 codes of q * 4, q_scale 1/4" if args.q_fp8 else "bf16",
            "mma": "e4m3 x e4m3 -> f32 tcgen05 (attend, two-term split), bf16 -> f32 tcgen05 (W_UV, both merge routes)",
            "launches_per_step": "attend, merge+value/gate" if not args.three_call else "attend, merge, value/gate",
            "timing": "value: CUDA-graph replay of the step; kernels_us / roofline: eager launches, one event pair each",
        },
        "kernels_us": step.kernels_us(t_att, t_mrg, t_val),
        "kv_tokens_per_s": step.stats["kv_tokens"] * args.steps * ws / total,
        "roofline": step.roofline(t_att),
        "e2e": {"value": aggregate_value(S, args.steps, ws, e2e_total), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "output_matches_device": bool(ok),
                "pipeline": "two steps in flight: step k+1's upload overlaps step k's kernels, read-back on a "
                            "second copy stream; buffers alternate between two sets",
                "l2": "not flushed between the overlapped steps: the default workload's KV rows (2.8 GB) exceed L2; "
                      "on workloads whose KV fits L2 partly, e2e runs L2-warm and can exceed the flushed value"},
        "gpu_launches": (3 if args.three_call else 2) * args.steps,
        "extra_ops": extra,
        "clocks": clk,
    }
    if per_workload:
        rec["per_workload"] = per_workload
    if ws == 1 and not args.no_cpu_baseline:
        rec["cpu_baseline"], rec["parity_check"] = cpu_baseline(spec, inp, gpu_out=gpu_out, one_thread=True,
                                                                q_fp8=args.q_fp8, causal=args.causal,
                                                                page_size=args.page_size)
    return rec


def _time_kv_append(S, k_scale, flush, dev, stream, warmup, steps):
    """The cache write of new tokens (not part of the timed step), into a
    pool of its own (the step's cache is left as it was): one new token per
    query row (decode), and a 65,536-token batch (bandwidth)."""
    res = {}
    pool = 1 << 17
    kv = torch.zeros((pool, 576), dtype=torch.uint8, device=dev)
    g = torch.Generator(device=dev).manual_seed(77)
    for name, T in (("decode_tokens", S), ("batch_65536", 65536)):
        kv_c = torch.randn(T, 512, generator=g, device=dev).to(torch.bfloat16)
        k_pe = torch.randn(T, 64, generator=g, device=dev).to(torch.bfloat16)
        slots = torch.randperm(pool, generator=g, device=dev)[:T].to(torch.int64)
        for _ in range(warmup):
            mla.kv_append(kv, kv_c, k_pe, slots, k_scale, stream=stream)
        ts = []
        for _ in range(steps):
            flush.fill_(1.0)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            mla.kv_append(kv, kv_c, k_pe, slots, k_scale, stream=stream)
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


def _host_cpu():
    """The host's CPU model (lscpu, else /proc/cpuinfo), core count and OpenMP setting."""
    model = None
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            k, _, v = line.partition(":")
            if k.strip() == "Model name" and v.strip():
                model = v.strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None and os.path.exists("/proc/cpuinfo"):
        for line in open("/proc/cpuinfo"):
            k, _, v = line.partition(":")
            if k.strip().lower() in ("model name", "cpu model") and v.strip():
                model = v.strip()
                break
    return {"cpu_model": model, "nproc": os.cpu_count(), "omp_num_threads": os.environ.get("OMP_NUM_THREADS")}


def _oracle_inputs(inp):
    """The step's inputs as the C oracle takes them (raw codes and bits)."""
    return dict(q=inp.q.cpu().contiguous().view(torch.int16).numpy().view(np.uint16), kv=inp.kv.cpu().numpy(),
                pages=inp.pages.cpu().numpy(), indptr=inp.indptr.cpu().numpy(),
                w=inp.w_uv.cpu().contiguous().view(torch.int16).numpy().view(np.uint16),
                g=inp.gate.cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _time_oracle(oracle, spec, inp, a, budget_s, threads=0):
    """Tokens/s of the C oracle over the whole workload, from a bounded
    sample: requests taken in a seeded random order (a request whose cost
    alone would take half the budget is passed over) until their estimated
    cost fills about budget_s on the host's threads, timed and repeated
    until about the budget is spent, then scaled to the workload by KV
    tokens (the oracle's work per request is proportional to its context
    length at fixed rows per request).  Returns (value, threads, sample
    text, sampled requests, the oracle's outputs)."""
    lens = np.diff(a["indptr"]).astype(np.int64)
    R = len(lens)
    nthreads = threads if threads > 0 else oracle.load_c().mla_oracle_threads()
    nz = np.nonzero(lens > 0)[0]
    probe_r = int(nz[np.argmin(lens[nz])]) if nz.size else 0
    t0 = time.perf_counter()
    oracle.decode_step_c(a["q"], a["kv"], a["pages"], a["indptr"], inp.scale, inp.kv_scale, spec.heads, spec.qlen,
                         a["w"], a["g"], requests=[probe_r], threads=threads)
    per_token = max(time.perf_counter() - t0, 1e-5) / max(1, lens[probe_r])
    order = np.random.default_rng(spec.seed).permutation(R)
    reqs, cost = [], 0.0
    for r in order:
        c = per_token * lens[r]
        if c > 0.5 * budget_s:
            continue
        if reqs and (cost + c) / max(1, min(nthreads, len(reqs) + 1)) > budget_s:
            break
        reqs.append(int(r))
        cost += c
    if not reqs:
        reqs = [probe_r]
    reqs.sort()
    reps, t0 = 0, time.perf_counter()
    while True:
        res = oracle.decode_step_c(a["q"], a["kv"], a["pages"], a["indptr"], inp.scale, inp.kv_scale, spec.heads,
                                   spec.qlen, a["w"], a["g"], requests=reqs, threads=threads)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s or dt / reps * (reps + 1) > 2 * budget_s:
            break
    tok_sample = int(lens[reqs].sum())
    tok_all = int(lens.sum())
    t_all = dt / reps * (tok_all / tok_sample if tok_sample > 0 else 1.0)
    sample = ("%d of %d requests (%d of %d KV tokens, seeded random order) x %d repetitions, full path in fp64 C, "
              "%.2f s; scaled to the whole workload by KV tokens" % (len(reqs), R, tok_sample, tok_all, reps, dt))
    return R * spec.qlen / t_all, int(nthreads), sample, reqs, res


def cpu_baseline(spec, inp, budget_s=10.0, gpu_out=None, one_thread=False, q_fp8=False, causal=False,
                 page_size=1):
    """Time the plain C fp64 oracle on the host cores on a bounded sample of
    the workload's requests (the first requests until ~budget_s of work).
    With ``gpu_out`` (out, latent, merged LSE of the timed GPU step, on the
    CPU) also returns the comparison of those rows with the oracle's; with
    ``one_thread`` also times one thread on the tiny and the single-token
    workloads."""
    import oracle  # test infrastructure: timed here as the CPU baseline only
    a = _oracle_inputs(inp)
    value, threads, sample, reqs, res = _time_oracle(oracle, spec, inp, a, budget_s)
    rec = {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample,
           "host": _host_cpu(), "build": "gcc -O2 -fopenmp (portable flags, no -march=native)"}
    if one_thread:
        rec["one_thread"] = {}
        for idx, budget in ((0, 2.0), (1, 5.0)):
            sp = W.WORKLOADS[idx]
            si = W.make_inputs(sp, "cpu")
            v, _, smp, _, _ = _time_oracle(oracle, sp, si, _oracle_inputs(si), budget, threads=1)
            rec["one_thread"][sp.name] = {"value": v, "unit": UNIT, "sample": smp}
    check = None
    if gpu_out is not None:
        if q_fp8 or causal or page_size != 1:
            check = {"skipped": "the C oracle covers the default step (bf16 query, no mask, page size 1)"}
        else:
            rlat, rlse, rout = res
            rows = np.concatenate([np.arange(r * spec.qlen, (r + 1) * spec.qlen) for r in reqs])
            g_out, g_lat, g_lse = (t.float().numpy().astype(np.float64)[rows] for t in gpu_out)
            r_out, r_lat, r_lse = rout[rows], rlat[rows], rlse[rows]
            err_out = np.abs(g_out - r_out)
            err_lat = np.abs(g_lat - r_lat)
            fin = np.isfinite(r_lse)
            same_inf = bool(np.array_equal(np.isneginf(g_lse), np.isneginf(r_lse)))
            lse_err = float(np.abs(g_lse[fin] - r_lse[fin]).max()) if fin.any() else 0.0
            ok_out = bool((err_out <= 2e-2 + 2e-2 * np.abs(r_out)).all())
            ok_lat = bool((err_lat <= 2e-2 + 2e-2 * np.abs(r_lat)).all())
            scale_out = float(err_out.max() / max(np.abs(r_out).max(), 1e-300))
            check = {"requests": len(reqs), "rows": int(len(rows)), "max_abs_err_out": float(err_out.max()),
                     "max_err_over_max_ref_out": scale_out, "max_abs_err_latent": float(err_lat.max()),
                     "max_abs_err_lse": lse_err,
                     "pass": ok_out and ok_lat and same_inf and lse_err <= 1e-3 and scale_out <= 2e-2,
                     "tolerance": "out / latent |err| <= 2e-2 + 2e-2 |ref| and max|err|/max|ref| <= 2e-2; LSE 1e-3"}
    return rec, check


def run_reference(args):
    ws, rank, local = _dist()
    if rank != 0:
        return None
    spec = _spec(args.workload, args.requests)
    inp = W.make_inputs(spec, "cpu")
    times = []
    base = None
    for k in range(args.warmup + args.steps):
        res, _ = cpu_baseline(spec, inp, budget_s=args.ref_budget)
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
                         "sample": base["sample"], "host": base["host"]},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="time the chosen workload only (not the other full-size workloads)")
    ap.add_argument("--three-call", action="store_true",
                    help="time merge and value/gate as two launches instead of the fused one")
    ap.add_argument("--ref-budget", type=float, default=5.0)
    ap.add_argument("--page-size", type=int, default=1,
                    help="KV cache as block tables of this many rows per block (power of two)")
    ap.add_argument("--q-fp8", action="store_true",
                    help="fp8 e4m3 query codes (q * 4) with q_scale 1/4 instead of the bf16 query")
    ap.add_argument("--no-plan", action="store_true",
                    help="round-robin work units under the split rule instead of the host work plan")
    ap.add_argument("--splits", default=None, metavar="NS:ST",
                    help="num_splits:split_tokens under the split rule (no work plan) instead of the host plan")
    ap.add_argument("--plan-splits", default=None, metavar="MIN:MAX",
                    help="host plan with at least MIN and at most MAX splits per request")
    ap.add_argument("--requests", type=int, default=None,
                    help="a smaller case of the workload: its first N requests (for profiling captures)")
    ap.add_argument("--causal", action="store_true",
                    help="causal mask within a request (row tq sees its first L - qlen + tq + 1 tokens)")
    ap.add_argument("--clocks-dir", default=None,
                    help="where the raw nvidia-smi clock samples go (default: the system temp directory)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.requests is not None and args.requests < 1:
        raise SystemExit("--requests must be at least 1")
    rec = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if rec is not None:
        print(json.dumps(rec), flush=True)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1 and args.impl != "reference":
        import torch.distributed as dist
        dist.destroy_process_group()
    if rec is not None and rec.get("parity_check") and rec["parity_check"].get("pass") is False:
        raise SystemExit(3)


if __name__ == "__main__":
    main()
