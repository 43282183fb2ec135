#!/usr/bin/env python3
"""Benchmark of the joint text/image attention hot path (QK-RMSNorm + RoPE
prologue, then joint attention) on one B300 per rank.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Metric: joint-attention TFLOP/s = 4 B H N^2 d / step time, on the FLUX-dev
1024x1024 step (B=1, H=24, d=128, 512 text + 64x64 image tokens, N=4608),
seeded synthetic bf16 inputs already resident in HBM.  A step is one
flux_attn_prologue + one flux_attn_attend call (= flux_attn_forward); L2 is
flushed (a 256 MB write) before every timed step, outside the step's events.
The FLUX 2048x2048 step (N=16896, BF16), the image-to-image step with a
2048x2048 reference image (N=33280, BF16) and the FP8 classifier-free-guidance
pair at 2048x2048 (B=2, N=16896: amax + E4M3 quantise + FP8 attention) are
measured the same way and reported under "secondary"; the QKV projection
with its fused QK-norm + RoPE epilogue (2 M F D flops: M = B N tokens,
F = 3 H 128 features, D = H 128 hidden) is reported under "qkv_projection".

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
import diffusion_transformer_joint_txt_b300 as fa  # noqa: E402

PRIMARY = "flux_1024_4608"
SECONDARY = ["flux_2048_16896", "i2i_2048_33280", "fp8_cfg_2048_16896", "vc_fp8_cfg_2048_16896",
             "sol_flux_2048_16896"]
METRIC = "joint-attn TFLOP/s & % of B300 BF16/FP8 TC peak at 4608/16896 tokens"
FALLBACK_PEAKS = {"bf16_tflops": 1800.0, "hbm_gbs": 6400.0}
L2_FLUSH_BYTES = 256 << 20
ATTN_SOURCES = ["diffusion_transformer_joint_txt_b300/csrc/attention.cuh",
                "diffusion_transformer_joint_txt_b300/csrc/ptx.cuh"]
# Dense per-GPU tensor-core figures the pages print (WaveSpeedAI X DataCrunch
# B200 page, technical-specifications table, without sparsity): context for
# the "frac_of_nominal" keys, not the roofline denominators.
NOMINAL_TFLOPS = {"bf16": 2250.0, "fp8": 4500.0}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(values, world, dist, torch, device):
    """Element-wise max of per-rank timings (the slowest rank decides); the
    identity on one rank.  `device` is "cuda" under NCCL, "cpu" under gloo."""
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(flops_per_rank, world, ms):
    """Whole-job TFLOP/s: every rank runs its own replica of the workload."""
    return flops_per_rank * world / (ms * 1e-3) / 1e12


def workload_config(w, world):
    """The "config" object of a JSON line; both arms print the same one."""
    return {"workload": w.name, "batch": w.batch, "heads": w.heads, "head_dim": 128,
            "tokens": w.tokens, "txt_len": w.txt_len, "img": [w.img_h, w.img_w],
            "ref": [w.ref_h, w.ref_w], "global_batch": w.batch * world, "seq_len": w.tokens,
            "parallelism": "replicas" if world > 1 else "single",
            "l2": "GPU arm: L2 flushed before every timed step (256 MB write, outside the step events)"}


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
                                          "--format=csv,noheader,nounits", "-lms", "20"],
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

    def summary(self, first=0, last=None):
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines[first:last]:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                pw.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "power_w": statistics.median(pw),
                "reasons": sorted(reasons), "samples": len(sm)}


def device_inputs(w, torch):
    inp = synthetic.make_inputs(w)
    dev = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda()
    return inp, dev(inp.q), dev(inp.k), dev(inp.v), torch.from_numpy(inp.w_q).cuda(), \
        torch.from_numpy(inp.w_k).cuda()


class Step:
    """One pass of the hot path over one workload, inputs resident in HBM:
    the prologue call, then the attention call, each bracketed by CUDA events
    on the launching stream."""

    def __init__(self, w, torch, fa):
        self.w = w
        self.fp8 = w.precision == "fp8"
        self.inp, self.q, self.k, self.v, self.wq, self.wk = device_inputs(w, torch)
        n = w.tokens
        self.attn = fa.FluxAttention(w.batch, w.heads, n, precision=w.precision,
                                     vc_repair_budget=w.vc_repair_budget, sol_tau=w.sol_tau)
        self.vc = w.vc_repair_budget > 0
        self.sol = w.sol_tau > 0
        if self.sol:
            nb = (n + 127) // 128
            self.keep = torch.empty((w.batch, w.heads, nb, nb), dtype=torch.uint8, device="cuda")
        self.geo = (w.txt_len, w.img_h, w.img_w, w.ref_h, w.ref_w)
        B, H = w.batch, w.heads
        if self.vc:
            R = self.attn.vc_repair_count(n)
            self.repair_idx = torch.empty((B, H, R), dtype=torch.int32, device="cuda")
            self.k_rep = torch.empty((B, H, R, 128), dtype=torch.bfloat16, device="cuda")
            self.v_rep = torch.empty_like(self.k_rep)
        if self.fp8:
            self.q8 = torch.empty((B, H, n, 128), dtype=torch.uint8, device="cuda")
            self.k8 = torch.empty_like(self.q8)
            self.v8t = torch.empty((B, H, 128, fa.pad16(n)), dtype=torch.uint8, device="cuda")
            self.scales = torch.empty((B, H, 3), dtype=torch.float32, device="cuda")
        else:
            self.qn = torch.empty((B, H, n, 128), dtype=torch.bfloat16, device="cuda")
            self.kn = torch.empty_like(self.qn)
        self.out = torch.empty_like(self.q)
        self.stream = torch.cuda.current_stream()

    def prologue(self):
        if self.vc:
            fa.flux_attn_prologue_fp8_vc(self.attn.handle, self.q, self.k, self.v, *self.geo, None, self.wq, self.wk,
                                         self.q8, self.k8, self.v8t, self.scales, self.repair_idx, self.k_rep,
                                         self.v_rep)
        elif self.fp8:
            self.attn.prologue_fp8(self.q, self.k, self.v, *self.geo, self.wq, self.wk, q8=self.q8, k8=self.k8,
                                   v8t=self.v8t, scales=self.scales)
        else:
            self.attn.prologue(self.q, self.k, *self.geo, self.wq, self.wk, qn=self.qn, kn=self.kn)
            if self.sol:   # the block mask is part of the sparse step's front half
                fa.flux_attn_sol_mask(self.attn.handle, self.qn, self.kn, self.w.tokens, self.keep)

    def attend(self):
        if self.vc:
            fa.flux_attn_attend_fp8_vc(self.attn.handle, self.q8, self.k8, self.v8t, self.scales, self.k_rep,
                                       self.v_rep, self.w.tokens, self.out)
        elif self.fp8:
            self.attn.attend_fp8(self.q8, self.k8, self.v8t, self.scales, out=self.out)
        elif self.sol:
            fa.flux_attn_attend_sol(self.attn.handle, self.qn, self.kn, self.v, self.keep, self.w.tokens, self.out)
        else:
            self.attn.attend(self.qn, self.kn, self.v, out=self.out)

    def processed_fraction(self):
        """Sparse steps: the share of the dense (query tile pair, key block) work
        the attention kernel does -- each CTA walks the union of the key blocks
        its two query tiles keep (1 for dense steps)."""
        if not self.sol:
            return 1.0, 1.0
        keep = self.keep.cpu().numpy().astype(bool)
        nb = keep.shape[-1]
        if nb % 2:
            keep = np.concatenate([keep, np.zeros(keep.shape[:2] + (1, nb), bool)], axis=2)
        union = keep[:, :, 0::2] | keep[:, :, 1::2]
        return float(union.mean()), float(keep[:, :, :nb].mean())

    def __call__(self, ev=None):
        """One step; ev = (start, end) brackets it, ev = (start, split, end)
        also splits it between the two calls."""
        if ev is not None:
            ev[0].record(self.stream)
        self.prologue()
        if ev is not None and len(ev) == 3:
            ev[1].record(self.stream)
        self.attend()
        if ev is not None:
            ev[-1].record(self.stream)

    @property
    def prologue_bytes(self):
        """Algorithmic HBM bytes of the prologue per step.  BF16: read q, k and
        write Q', K' (2 + 2 bytes per element each).  FP8: per element of each
        of Q', K', V, one bf16 read and one E4M3 byte written (3 bytes, so 9 per
        (b, n, h, d): 934 MB on the CFG pair), the figure the hot-path scope
        fixes for this step."""
        elems = self.w.batch * self.w.tokens * self.w.heads * 128
        return elems * (9 if self.fp8 else 8)

    @property
    def prologue_traffic_min(self):
        """Bytes the prologue cannot avoid moving.  FP8: the scales need the
        amax of a whole head first, so q, k, v are read twice (2 x 6 bytes)
        around the three code bytes: 15 bytes per (b, n, h, d)."""
        elems = self.w.batch * self.w.tokens * self.w.heads * 128
        return elems * (15 if self.fp8 else 8)


class QKVStep:
    """The QKV projection with its fused QK-norm + RoPE epilogue over one
    workload (hidden size H * 128), inputs resident in HBM."""

    def __init__(self, w, torch, fa):
        self.w = w
        inp = synthetic.make_qkv_inputs(w)
        dev = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda()
        self.x, self.wt = dev(inp.x), dev(inp.w)
        self.bias = torch.from_numpy(inp.bias).cuda()
        self.wq, self.wk = torch.from_numpy(inp.w_q).cuda(), torch.from_numpy(inp.w_k).cuda()
        self.fp8 = w.precision == "fp8"
        self.attn = fa.FluxAttention(w.batch, w.heads, w.tokens, precision=w.precision)
        n, B, H = w.tokens, w.batch, w.heads
        if self.fp8:   # the codes the FP8 attention reads
            self.q8 = torch.empty((B, H, n, 128), dtype=torch.uint8, device="cuda")
            self.k8 = torch.empty_like(self.q8)
            self.v8t = torch.empty((B, H, 128, fa.pad16(n)), dtype=torch.uint8, device="cuda")
            self.scales = torch.empty((B, H, 3), dtype=torch.float32, device="cuda")
        else:
            self.qn = torch.empty((B, H, n, 128), dtype=torch.bfloat16, device="cuda")
            self.kn = torch.empty_like(self.qn)
            self.v = torch.empty((B, n, H, 128), dtype=torch.bfloat16, device="cuda")
        self.stream = torch.cuda.current_stream()
        self.flops = 2 * B * n * (3 * H * 128) * inp.d_model

    def __call__(self, ev=None):
        if ev is not None:
            ev[0].record(self.stream)
        geo = (self.w.txt_len, self.w.img_h, self.w.img_w, self.w.ref_h, self.w.ref_w)
        if self.fp8:
            fa.flux_attn_qkv_fp8(self.attn.handle, self.x, self.wt, self.bias, self.x.shape[-1], *geo, None, self.wq,
                                 self.wk, self.q8, self.k8, self.v8t, self.scales)
        else:
            self.attn.qkv(self.x, self.wt, self.bias, *geo, self.wq, self.wk, qn=self.qn, kn=self.kn, v=self.v)
        if ev is not None:
            for e in ev[1:]:
                e.record(self.stream)


def sustained(step, seconds, torch, clocks):
    """The attention kernel back to back for about `seconds` (no L2 flush):
    the power-limited steady state, with the clocks and power of that window."""
    for _ in range(5):
        step.attend()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    step.attend()
    torch.cuda.synchronize()
    reps = max(10, int(seconds / max(time.perf_counter() - t0, 1e-5)))
    first = len(clocks.lines)
    e0.record(step.stream)
    for _ in range(reps):
        step.attend()
    e1.record(step.stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    if step.attn.sync_status() != 0:
        raise RuntimeError("device status error in the sustained run (%s)" % step.w.name)
    return ms, reps, clocks.summary(first, len(clocks.lines))


def measure(step, steps, warmup, torch, flush, barrier):
    """Mean step, attention-kernel and prologue times (ms) over `steps` timed
    steps, from three CUDA events per step on the launching stream (before the
    prologue, between the two calls, after the attention); L2 is flushed
    before every step, outside its events."""
    for _ in range(warmup):
        flush.zero_()
        step()
    if step.attn.sync_status() != 0:
        raise RuntimeError("device status error in warm-up (%s)" % step.w.name)
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    barrier()
    for e in ev:
        flush.zero_()
        step(e)
    barrier()
    if step.attn.sync_status() != 0:
        raise RuntimeError("device status error during the timed region (%s)" % step.w.name)
    return (sum(a.elapsed_time(c) for a, _, c in ev) / steps,
            sum(b.elapsed_time(c) for _, b, c in ev) / steps,
            sum(a.elapsed_time(b) for a, b, _ in ev) / steps)


def run_ours(args):
    import torch
    import torch.distributed as dist
    import diffusion_transformer_joint_txt_b300 as fa

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    peaks, peak_kind = load_peaks()
    peak_bf16 = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def slowest(vals):
        return max_over_ranks(vals, world, dist, torch, "cuda")

    def summary(step, times, n_steps):
        w = step.w
        s_ms, a_ms, p_ms = times
        peak = peak_bf16 * (2.0 if step.fp8 else 1.0)
        nominal = NOMINAL_TFLOPS["fp8" if step.fp8 else "bf16"]
        achieved = w.flops / (a_ms * 1e-3) / 1e12
        extra = {}
        if step.sol:
            processed, kept = step.processed_fraction()
            # dense-equivalent rate as "attn_tflops"; the roofline counts the work done
            extra = {"sol_tau": w.sol_tau, "kept_block_fraction": kept, "processed_fraction": processed,
                     "attn_tflops_processed": achieved * processed}
            achieved_roof = achieved * processed
        else:
            achieved_roof = achieved
        return {**extra, "workload": w.name, "precision": w.precision, "batch": w.batch, "heads": w.heads,
                "tokens": w.tokens, "steps": n_steps, "value": job_throughput(w.flops, world, s_ms),
                "ms_per_step": s_ms, "attn_kernel_ms": a_ms, "attn_tflops": achieved,
                "roofline_frac": achieved_roof / peak, "peak_tflops": peak,
                "frac_of_nominal": achieved / nominal, "nominal_tflops": nominal,
                "prologue_ms": p_ms, "prologue_gbs": step.prologue_bytes / (p_ms * 1e-3) / 1e9,
                "prologue_frac": step.prologue_bytes / (p_ms * 1e-3) / 1e9 / hbm,
                "prologue_algorithmic_bytes": step.prologue_bytes,
                "prologue_traffic_min_gbs": step.prologue_traffic_min / (p_ms * 1e-3) / 1e9,
                "gpu_launches": n_steps * step.attn.launches_per_forward(w.tokens)}

    w = synthetic.WORKLOADS[args.workload]
    main_step = Step(w, torch, fa)
    others = [] if args.no_secondary else [Step(synthetic.WORKLOADS[n], torch, fa) for n in args.secondary]
    with ClockSampler(local) as clocks:
        t0 = time.perf_counter()
        c0 = len(clocks.lines)
        times = slowest(list(measure(main_step, args.steps, args.warmup, torch, flush, barrier)))
        c1 = len(clocks.lines)
        wall = time.perf_counter() - t0
        other_times = [slowest(list(measure(st, args.steps2, args.warmup, torch, flush, barrier)))
                       for st in others]
        sus = []
        if args.sustained_seconds > 0:
            for st in [main_step] + [o for o in others if o.w.precision == "bf16" and not o.sol]:
                ms_s, reps_s, clk_s = sustained(st, args.sustained_seconds, torch, clocks)
                sus.append((st, ms_s, reps_s, clk_s))
        qkv_steps = [] if args.no_secondary else [QKVStep(synthetic.WORKLOADS[n], torch, fa) for n in args.qkv]
        qkv_times = [slowest(list(measure(st, args.steps2, args.warmup, torch, flush, barrier)))
                     for st in qkv_steps]
    main = summary(main_step, times, args.steps)
    secondary = [summary(st, t, args.steps2) for st, t in zip(others, other_times)]
    peak_sus = float(peaks.get("bf16_tflops_sustained", 0.0)) or None
    sustained_lines = []
    for st, ms_s, reps_s, clk_s in sus:
        tf = st.w.flops / (ms_s * 1e-3) / 1e12
        sustained_lines.append({"workload": st.w.name, "kernel": "attn_kernel<bf16>", "launches": reps_s, "ms": ms_s,
                                "achieved": tf, "peak": peak_sus, "unit": "TFLOP/s",
                                "frac": tf / peak_sus if peak_sus else None,
                                "peak_kind": peak_kind + " bf16 sustained", "clocks": clk_s})
    qkv = []
    for st, (s_ms, _, _) in zip(qkv_steps, qkv_times):
        # one call = the (cos, sin) table kernel + the GEMM; both are in the time
        tf = st.flops / (s_ms * 1e-3) / 1e12
        kern = "qkv_gemm_kernel (+ rope_table_kernel)" + (" + E4M3 codes (fp8_vt_kernel, fp8_codes_kernel)"
                                                           if st.fp8 else "")
        qkv.append({"workload": st.w.name, "precision": st.w.precision, "kernel": kern,
                    "gemm": [st.w.batch * st.w.tokens, 3 * st.w.heads * 128, st.w.heads * 128],
                    "ms": s_ms, "tflops": tf, "roofline_frac": tf / peak_bf16, "frac_of_2250_nominal": tf / NOMINAL_TFLOPS["bf16"],
                    "algorithmic_flops": st.flops, "gpu_launches": (4 if st.fp8 else 2) * args.steps2})
        st.attn.close()

    # end to end through the public API: pinned host inputs in, result back out, every step
    e2e = run_e2e(w, main_step.inp, main_step.attn, torch, args.e2e_steps, world, dist)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, main_step.inp, args.cpu_seconds)

    line = {
        "metric": METRIC, "value": main["value"], "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": main["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, norm weights 1+0.1N(0,1))",
        "config": workload_config(w, world),
        "roofline": {"bound": "tensor", "kernel": "attn_kernel<bf16>", "achieved": main["attn_tflops"],
                     "peak": peak_bf16, "unit": "TFLOP/s", "frac": main["roofline_frac"],
                     "peak_kind": peak_kind + " bf16 burst", "frac_of_2250_nominal": main["frac_of_nominal"],
                     "traffic": ncu_traffic(w.name), "algorithmic_flops_per_launch": w.flops},
        "prologue": {"ms": main["prologue_ms"], "gbs": main["prologue_gbs"], "hbm_peak_gbs": hbm,
                     "frac": main["prologue_gbs"] / hbm, "algorithmic_bytes": main_step.prologue_bytes},
        "attn_kernel_ms": main["attn_kernel_ms"],
        "e2e": e2e,
        "gpu_launches": main["gpu_launches"],
        "clocks": clocks.summary(c0, c1),
        "wall_s_timed_region": wall,
        "cpu_baseline": cpu,
        "secondary": secondary,
        "qkv_projection": qkv,
        "roofline_sustained": sustained_lines,
    }
    for st in [main_step] + others:
        st.attn.close()
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(w, inp, attn, torch, steps, world, dist):
    """Same metric through FluxAttention.forward with pinned host buffers:
    every step copies q, k, v and the norm weights in and the output back
    out.  Steps are pipelined over two sets of device buffers on three
    streams -- step i+1's inputs travel host -> device while step i computes
    and step i-1's output travels back -- and the timed region runs from the
    first input copy to the last output copy."""
    host = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).pin_memory()
    hq, hk, hv = host(inp.q), host(inp.k), host(inp.v)
    hwq = torch.from_numpy(inp.w_q).pin_memory()
    hwk = torch.from_numpy(inp.w_k).pin_memory()
    hins = (hq, hk, hv, hwq, hwk)
    houts = [torch.empty_like(hq).pin_memory() for _ in range(2)]
    sets = [[torch.empty_like(t, device="cuda") for t in hins] + [torch.empty_like(hq, device="cuda")]
            for _ in range(2)]
    h2d_s, comp_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    loaded, computed, drained = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    geo = (w.txt_len, w.img_h, w.img_w, w.ref_h, w.ref_w)

    def run(n):
        for i in range(n):
            s = i % 2
            dq, dk, dv, dwq, dwk, dout = sets[s]
            with torch.cuda.stream(h2d_s):
                if i >= 2:
                    h2d_s.wait_event(computed[s])          # step i-2 is done with these inputs
                for d, h in zip(sets[s][:5], hins):
                    d.copy_(h, non_blocking=True)
                loaded[s].record(h2d_s)
            with torch.cuda.stream(comp_s):
                comp_s.wait_event(loaded[s])
                if i >= 2:
                    comp_s.wait_event(drained[s])          # step i-2's output has left dout
                attn.forward(dq, dk, dv, *geo, dwq, dwk, out=dout, stream=comp_s)
                computed[s].record(comp_s)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(computed[s])
                houts[s].copy_(dout, non_blocking=True)
                drained[s].record(d2h_s)

    run(2)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(h2d_s)
    run(steps)
    e1.record(d2h_s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    ms = max_over_ranks([ms], world, dist, torch, "cuda")[0]
    h2d = sum(t.numel() * t.element_size() for t in hins)
    d2h = houts[0].numel() * houts[0].element_size()
    return {"value": job_throughput(w.flops, world, ms), "unit": "TFLOP/s", "ms_per_step": ms,
            "steps": steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelined": "2 buffer sets, H2D / compute / D2H on separate streams",
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

    # grow the sample until it takes a meaningful share of `seconds`, then size
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
        "config": workload_config(w, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=PRIMARY, choices=sorted(synthetic.WORKLOADS))
    ap.add_argument("--steps2", type=int, default=60, help="timed steps of each secondary workload")
    ap.add_argument("--secondary", nargs="*", default=SECONDARY, choices=sorted(synthetic.WORKLOADS),
                    help="workloads measured after the primary one and reported under \"secondary\"")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--sustained-seconds", type=float, default=2.0,
                    help="seconds of back-to-back attention launches per BF16 workload for the power-limited "
                         "steady state (0 skips)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--reference-rows", type=int, default=2048)
    ap.add_argument("--qkv", nargs="*", default=["flux_1024_4608", "flux_2048_16896", "fp8_cfg_2048_16896"],
                    choices=sorted(synthetic.WORKLOADS),
                    help="workloads whose QKV projection (fused QK-norm + RoPE epilogue) is measured")
    ap.add_argument("--no-secondary", action="store_true", help="measure the primary workload only")
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
