#!/usr/bin/env python3
"""Benchmark of the joint text/image attention hot path (QK-RMSNorm + RoPE
prologue, then joint attention) on one B300 per rank.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Metric: joint-attention TFLOP/s = 4 B H N^2 d / step time, on the FLUX-dev
1024x1024 step (B=1, H=24, d=128, 512 text + 64x64 image tokens, N=4608),
seeded synthetic bf16 inputs already resident in HBM.  A step is one
flux_attn_prologue + one flux_attn_attend call (= flux_attn_forward); L2 is
flushed (a 256 MB write) before every timed step, outside the step's events.
The FLUX 2048x2048 step (N=16896) is measured the same way and reported under
"secondary".

One JSON line on rank 0.  Under torchrun every rank runs its own replica of
the workload (the (batch, head) units are independent; no collective is on
the data path), a barrier brackets the timed region and the slowest rank's
time is used.

--impl reference times the fp64 CPU oracle on a bounded sample of query rows
of the same workload, on the host cores, and prints the same line with
"impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

PRIMARY = "flux_1024_4608"
SECONDARY = "flux_2048_16896"
METRIC = "joint-attn TFLOP/s & % of B300 BF16/FP8 TC peak at 4608/16896 tokens"
FALLBACK_PEAKS = {"bf16_tflops": 1800.0, "hbm_gbs": 6400.0}
L2_FLUSH_BYTES = 256 << 20
ATTN_SOURCES = ["diffusion_transformer_joint_txt_b300/csrc/attention_bf16.cuh",
                "diffusion_transformer_joint_txt_b300/csrc/ptx.cuh"]


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_sha(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """DRAM bytes per launch of the attention kernel from the committed ncu
    summary, or None when it is absent or the kernel changed since."""
    path = os.path.join(ROOT, "profiles", "attn_bf16_%s.traffic.json" % workload)
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("source_sha") != source_sha(ATTN_SOURCES):
        return None
    return t.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        time.sleep(0.15)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        # samples under load: the upper part of the distribution
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def device_inputs(w, torch):
    inp = synthetic.make_inputs(w)
    dev = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda()
    return inp, dev(inp.q), dev(inp.k), dev(inp.v), torch.from_numpy(inp.w_q).cuda(), \
        torch.from_numpy(inp.w_k).cuda()


def time_device(w, steps, warmup, torch, fa, flush):
    """Device-timed steps: returns (mean step ms, mean attention-kernel ms, launches, out)."""
    inp, q, k, v, wq, wk = device_inputs(w, torch)
    n = w.tokens
    attn = fa.FluxAttention(w.batch, w.heads, n)
    hm = (w.batch, w.heads, n, 128)
    qn = torch.empty(hm, dtype=torch.bfloat16, device="cuda")
    kn = torch.empty(hm, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream()
    geo = (w.txt_len, w.img_h, w.img_w, w.ref_h, w.ref_w)

    def step():
        attn.prologue(q, k, *geo, wq, wk, qn=qn, kn=kn)
        attn.attend(qn, kn, v, out=out)

    for _ in range(warmup):
        flush.zero_()
        step()
    if attn.sync_status() != 0:
        raise RuntimeError("device status error in warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    return attn, step, ev, (q, k, v, wq, wk, out, qn, kn), geo, inp, stream


def run_ours(args):
    import torch
    import torch.distributed as dist
    import diffusion_transformer_joint_txt_b300 as fa

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    peaks, peak_kind = load_peaks()
    w = synthetic.WORKLOADS[args.workload]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    attn, step, ev, bufs, geo, inp, stream = time_device(w, args.steps, args.warmup, torch, fa, flush)
    q, k, v, wq, wk, out, qn, kn = bufs

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    with ClockSampler(local) as clocks:
        barrier()
        t0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            e0, e1, e2 = ev[i]
            e0.record(stream)
            attn.prologue(q, k, *geo, wq, wk, qn=qn, kn=kn)
            e1.record(stream)
            attn.attend(qn, kn, v, out=out)
            e2.record(stream)
        barrier()
        wall = time.perf_counter() - t0
    status = attn.sync_status()
    if status != 0:
        raise RuntimeError("device status %d during the timed region" % status)
    step_ms = sum(a.elapsed_time(c) for a, _, c in ev) / args.steps
    attn_ms = sum(b.elapsed_time(c) for _, b, c in ev) / args.steps
    pro_ms = sum(a.elapsed_time(b) for a, b, _ in ev) / args.steps
    launches = args.steps * attn.launches_per_forward(w.tokens)

    # slowest rank decides
    t = torch.tensor([step_ms, attn_ms, pro_ms], dtype=torch.float64, device="cuda")
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    step_ms, attn_ms, pro_ms = t.tolist()

    flops = w.flops
    value = flops * world / (step_ms * 1e-3) / 1e12
    achieved = flops / (attn_ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    pro_bytes = 4 * w.batch * w.tokens * w.heads * 128 * 2      # read q, k; write q', k'
    traffic = ncu_traffic(w.name)

    # end to end through the public API: pinned host inputs in, result back out, every step
    e2e = run_e2e(w, inp, attn, torch, args.e2e_steps, world, dist)

    secondary = None
    if not args.no_secondary:
        attn2, step2, ev2, bufs2, geo2, _, _ = time_device(synthetic.WORKLOADS[SECONDARY], args.steps2,
                                                           args.warmup, torch, fa, flush)
        q2, k2, v2, wq2, wk2, out2, qn2, kn2 = bufs2
        barrier()
        for i in range(args.steps2):
            flush.zero_()
            e0, e1, e2 = ev2[i]
            e0.record(stream)
            attn2.prologue(q2, k2, *geo2, wq2, wk2, qn=qn2, kn=kn2)
            e1.record(stream)
            attn2.attend(qn2, kn2, v2, out=out2)
            e2.record(stream)
        barrier()
        if attn2.sync_status() != 0:
            raise RuntimeError("device status error (secondary)")
        s_ms = sum(a.elapsed_time(c) for a, _, c in ev2) / args.steps2
        a_ms = sum(b.elapsed_time(c) for _, b, c in ev2) / args.steps2
        w2 = synthetic.WORKLOADS[SECONDARY]
        secondary = {"workload": SECONDARY, "tokens": w2.tokens, "steps": args.steps2,
                     "value": w2.flops / (s_ms * 1e-3) / 1e12, "ms_per_step": s_ms,
                     "attn_kernel_ms": a_ms, "attn_tflops": w2.flops / (a_ms * 1e-3) / 1e12,
                     "roofline_frac": w2.flops / (a_ms * 1e-3) / 1e12 / peak,
                     "frac_of_2250_nominal": w2.flops / (a_ms * 1e-3) / 1e12 / 2250.0}
        attn2.close()
        secondary["gpu_launches"] = args.steps2 * 2

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, inp, args.cpu_seconds)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, norm weights 1+0.1N(0,1))",
        "config": {"workload": w.name, "batch": w.batch, "heads": w.heads, "head_dim": 128,
                   "tokens": w.tokens, "txt_len": w.txt_len, "img": [w.img_h, w.img_w],
                   "global_batch": w.batch * world, "seq_len": w.tokens,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "flushed before every timed step (256 MB write, outside the step events)"},
        "roofline": {"bound": "tensor", "kernel": "attn_bf16_kernel", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "peak_kind": peak_kind + " bf16 burst",
                     "frac_of_2250_nominal": achieved / 2250.0, "traffic": traffic,
                     "algorithmic_flops_per_launch": flops},
        "prologue": {"ms": pro_ms, "gbs": pro_bytes / (pro_ms * 1e-3) / 1e9, "hbm_peak_gbs": hbm,
                     "frac": pro_bytes / (pro_ms * 1e-3) / 1e9 / hbm, "algorithmic_bytes": pro_bytes},
        "attn_kernel_ms": attn_ms,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks.summary(),
        "wall_s_timed_region": wall,
        "cpu_baseline": cpu,
        "secondary": secondary,
    }
    attn.close()
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(w, inp, attn, torch, steps, world, dist):
    """Same metric through FluxAttention.forward with pinned host buffers:
    every step copies q, k, v, the norm weights in, and the output back out."""
    host = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).pin_memory()
    hq, hk, hv = host(inp.q), host(inp.k), host(inp.v)
    hwq = torch.from_numpy(inp.w_q).pin_memory()
    hwk = torch.from_numpy(inp.w_k).pin_memory()
    hout = torch.empty_like(hq).pin_memory()
    dq, dk, dv = (torch.empty_like(t, device="cuda") for t in (hq, hk, hv))
    dwq, dwk = torch.empty_like(hwq, device="cuda"), torch.empty_like(hwk, device="cuda")
    dout = torch.empty_like(dq)
    stream = torch.cuda.current_stream()
    geo = (w.txt_len, w.img_h, w.img_w, w.ref_h, w.ref_w)

    def step():
        for d, h in ((dq, hq), (dk, hk), (dv, hv), (dwq, hwq), (dwk, hwk)):
            d.copy_(h, non_blocking=True)
        attn.forward(dq, dk, dv, *geo, dwq, dwk, out=dout)
        hout.copy_(dout, non_blocking=True)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    t = torch.tensor([ms], dtype=torch.float64, device="cuda")
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms = float(t.item())
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hwq, hwk))
    d2h = hout.numel() * hout.element_size()
    return {"value": w.flops * world / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "steps": steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "gpu_launches": steps * attn.launches_per_forward(w.tokens)}


def cpu_baseline(w, inp, seconds):
    """The oracle as it stands, timed on a bounded sample of query rows of the
    workload; TFLOP/s counts 4 N d flops per output row."""
    import oracle
    oracle.build()
    threads = oracle.max_threads()
    rng = np.random.default_rng(5)
    n = w.tokens
    per_row = 4.0 * n * 128

    def timed(count):
        rows = np.stack([np.zeros(count, np.int64), rng.integers(0, w.heads, count),
                         rng.integers(0, n, count)], 1)
        rows = rows[np.argsort(rows[:, 1], kind="stable")]
        t0 = time.perf_counter()
        oracle.attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k, rows=rows, nthreads=threads)
        return time.perf_counter() - t0

    # grow the sample until it takes a meaningful share of the budget, then size
    # the measured sample from that rate (per-head set-up makes tiny probes misleading)
    count, t = 256, 0.0
    while count < 400000:
        t = timed(count)
        if t >= seconds / 8:
            break
        count *= 4
    count = int(min(400000, max(count, count * seconds / max(t, 1e-6))))
    t = timed(count)
    return {"value": count * per_row / t / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": "%d query rows of %s (random heads), %.1f s, fp64 C + OpenMP" % (count, w.name, t),
            "seconds": t}


def run_reference(args):
    """The oracle arm: each step is a bounded sample of query rows."""
    rank, world, local = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = synthetic.WORKLOADS[args.workload]
    inp = synthetic.make_inputs(w)
    threads = oracle.max_threads()
    n = w.tokens
    per_row = 4.0 * n * 128
    rows_per_step = args.reference_rows
    rng = np.random.default_rng(9)

    def step():
        rows = np.stack([np.zeros(rows_per_step, np.int64), rng.integers(0, w.heads, rows_per_step),
                         rng.integers(0, n, rows_per_step)], 1)
        rows = rows[np.argsort(rows[:, 1], kind="stable")]
        oracle.attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k, rows=rows, nthreads=threads)

    for _ in range(args.warmup):
        step()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = rows_per_step * per_row / (ms * 1e-3) / 1e12
    sample = "%d query rows of %s per step (random heads), fp64 C + OpenMP" % (rows_per_step, w.name)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) bf16)", "impl": "reference",
        "config": {"workload": w.name, "batch": w.batch, "heads": w.heads, "head_dim": 128,
                   "tokens": w.tokens, "global_batch": w.batch, "seq_len": w.tokens},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=PRIMARY, choices=sorted(synthetic.WORKLOADS))
    ap.add_argument("--steps2", type=int, default=60, help="timed steps of the secondary workload")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--reference-rows", type=int, default=2048)
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
