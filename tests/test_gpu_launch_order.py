"""The attention kernel is launched as a programmatic dependent of the kernel
before it in the stream and waits for that grid before its first global
read.  These tests alternate two input sets step after step with no host
synchronisation (with and without an event recorded between the two calls)
and require every step's output to equal, bit for bit, the output of the
same inputs computed with a synchronisation between the prologue and the
attention: an attention that read Q', K' (or the FP8 codes) before the
prologue had finished would return the other set's result.
"""
import numpy as np
import pytest
import torch

import synthetic
from gpu_util import device_inputs

pytestmark = pytest.mark.gpu

import diffusion_transformer_joint_txt_b300 as fa  # noqa: E402

STEPS = 12


def _geom(w):
    return w.txt_len, w.img_h, w.img_w, w.ref_h, w.ref_w


def _alternating(w, run_prologue, run_attend, out):
    """run_prologue(i) for input set i % 2, then run_attend(); a snapshot of
    out per step; every fourth pair of steps records an event in between."""
    mid = torch.cuda.Event()
    snaps = torch.empty((STEPS,) + tuple(out.shape), dtype=out.dtype, device=out.device)
    for i in range(STEPS):
        run_prologue(i % 2)
        if i % 4 >= 2:
            mid.record()
        run_attend()
        snaps[i].copy_(out)
    torch.cuda.synchronize()
    return snaps


@pytest.mark.parametrize("precision", ["bf16", "fp8"])
def test_prologue_then_attention_no_sync(precision):
    w = synthetic.Workload("order", 1, 8, 512, 48, 64, 0, 0, precision=precision, outliers=False)  # N = 3584
    inp = synthetic.make_inputs(w, seed=21)
    d = device_inputs(inp)
    sets = [(d["q"], d["k"]), (torch.flip(d["q"], dims=[1]).contiguous(), (-d["k"]).contiguous())]
    attn = fa.FluxAttention(w.batch, w.heads, w.tokens, precision=precision)
    out = torch.empty_like(d["q"])
    geo = _geom(w)
    if precision == "fp8":
        bufs = attn.prologue_fp8(d["q"], d["k"], d["v"], *geo, d["q_norm_w"], d["k_norm_w"])

        def pro(s):
            attn.prologue_fp8(sets[s][0], sets[s][1], d["v"], *geo, d["q_norm_w"], d["k_norm_w"], q8=bufs[0],
                              k8=bufs[1], v8t=bufs[2], scales=bufs[3])

        def att():
            attn.attend_fp8(*bufs, out=out)
    else:
        bufs = attn.prologue(d["q"], d["k"], *geo, d["q_norm_w"], d["k_norm_w"])

        def pro(s):
            attn.prologue(sets[s][0], sets[s][1], *geo, d["q_norm_w"], d["k_norm_w"], qn=bufs[0], kn=bufs[1])

        def att():
            attn.attend(bufs[0], bufs[1], d["v"], out=out)
    refs = []
    for s in range(2):
        pro(s)
        torch.cuda.synchronize()
        att()
        torch.cuda.synchronize()
        refs.append(out.clone())
    assert not torch.equal(refs[0], refs[1])
    snaps = _alternating(w, pro, att, out)
    assert attn.sync_status() == 0
    bad = [i for i in range(STEPS) if not torch.equal(snaps[i], refs[i % 2])]
    assert not bad, "steps whose output is not their own inputs' result: %s" % bad


def test_forward_alternating_inputs():
    w = synthetic.Workload("order_fwd", 2, 4, 256, 32, 40, 8, 8, outliers=False)   # N = 1600, B = 2
    inp = synthetic.make_inputs(w, seed=22)
    d = device_inputs(inp)
    sets = [(d["q"], d["k"], d["v"]), (d["k"].clone(), d["q"].clone(), torch.flip(d["v"], dims=[1]).contiguous())]
    attn = fa.FluxAttention(w.batch, w.heads, w.tokens)
    out = torch.empty_like(d["q"])
    refs = []
    for s in sets:
        attn.forward(*s, *_geom(w), d["q_norm_w"], d["k_norm_w"], out=out)
        torch.cuda.synchronize()
        refs.append(out.clone())
    snaps = torch.empty((STEPS,) + tuple(out.shape), dtype=out.dtype, device=out.device)
    for i in range(STEPS):
        attn.forward(*sets[i % 2], *_geom(w), d["q_norm_w"], d["k_norm_w"], out=out)
        snaps[i].copy_(out)
    torch.cuda.synchronize()
    assert attn.sync_status() == 0
    assert all(torch.equal(snaps[i], refs[i % 2]) for i in range(STEPS))
