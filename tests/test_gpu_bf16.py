"""BF16 joint attention through the C ABI against the fp64 oracle (GPU).

Every row for the small cases; at the full FLUX sizes a seeded sample of rows
per (b, h) plus every stream and tile boundary row, and one whole head.
Tolerances (gpu_util): max-abs 1e-2, mean-abs 1e-3, relative RMS 1e-2.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import (BF16_MAX_ABS, BF16_MEAN_ABS, BF16_REL_RMS, compare, dev_bf16, device_inputs,
                      gather_rows, host_f64)

pytestmark = pytest.mark.gpu

import diffusion_transformer_joint_txt_b300 as fa  # noqa: E402


def _run(w, inp, use_pos=False, handle=None):
    d = device_inputs(inp)
    attn = handle or fa.FluxAttention(w.batch, w.heads, inp.pos.shape[0])
    n = inp.pos.shape[0]
    txt, ih, iw, rh, rw = _geom(w, n)
    out = attn.forward(d["q"], d["k"], d["v"], txt, ih, iw, rh, rw, d["q_norm_w"], d["k_norm_w"],
                       pos_ids=d["pos_ids"] if use_pos else None)
    assert attn.sync_status() == 0
    return out, attn


def _geom(w, n):
    return w.txt_len, w.img_h, w.img_w, w.ref_h, w.ref_w


def test_tiny_every_row():
    w = synthetic.WORKLOADS["tiny_320"]
    inp = synthetic.make_inputs(w)
    out, _ = _run(w, inp)
    want = oracle.attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k)
    compare(host_f64(out), want, BF16_MAX_ABS, BF16_MEAN_ABS, BF16_REL_RMS, "tiny_320")


@pytest.mark.parametrize("B,H,txt,ih,iw,rh,rw", [
    (2, 3, 5, 7, 9, 2, 3),        # 148 tokens: fewer chunks than SMs
    (2, 5, 17, 30, 40, 9, 11),    # 2632 tokens, odd H: every block walks several chunks of the ring
    (1, 24, 512, 16, 16, 0, 0),   # the FLUX head count, 768 tokens
])
def test_prologue_matches_oracle(B, H, txt, ih, iw, rh, rw):
    w = synthetic.Workload("prologue", B, H, txt, ih, iw, rh, rw)
    inp = synthetic.make_inputs(w)
    d = device_inputs(inp)
    n = inp.pos.shape[0]
    attn = fa.FluxAttention(w.batch, w.heads, n)
    qn, kn = attn.prologue(d["q"], d["k"], *_geom(w, n), d["q_norm_w"], d["k_norm_w"])
    assert attn.sync_status() == 0
    for got, x, wt in ((qn, inp.q, inp.w_q), (kn, inp.k, inp.w_k)):
        want = oracle.prologue(x, inp.pos, wt).transpose(0, 2, 1, 3)   # -> [B, H, N, d]
        g = host_f64(got)
        err = np.abs(g - want)
        # fp32 arithmetic, then one bf16 rounding (half an ulp = 2^-9 relative)
        assert np.all(err <= 2.0 ** -8 * np.abs(want) + 1e-5), float((err / (np.abs(want) + 1e-5)).max())


def test_explicit_positions_equal_generated_ones():
    w = synthetic.Workload("pos_check", 1, 2, 13, 9, 11, 4, 6)
    inp = synthetic.make_inputs(w)
    a, attn = _run(w, inp, use_pos=False)
    b, _ = _run(w, inp, use_pos=True, handle=attn)
    assert torch.equal(a, b)


def test_split_calls_equal_forward_and_are_deterministic():
    w = synthetic.WORKLOADS["tiny_320"]
    inp = synthetic.make_inputs(w)
    d = device_inputs(inp)
    n = inp.pos.shape[0]
    attn = fa.FluxAttention(w.batch, w.heads, n)
    full = attn.forward(d["q"], d["k"], d["v"], *_geom(w, n), d["q_norm_w"], d["k_norm_w"])
    qn, kn = attn.prologue(d["q"], d["k"], *_geom(w, n), d["q_norm_w"], d["k_norm_w"])
    split = attn.attend(qn, kn, d["v"])
    again = attn.forward(d["q"], d["k"], d["v"], *_geom(w, n), d["q_norm_w"], d["k_norm_w"])
    assert attn.sync_status() == 0
    assert torch.equal(full, split)
    assert torch.equal(full, again)


RAGGED = [
    (2, 3, 7, 5, 9, 0, 0),        # N = 52, one partial tile
    (1, 2, 0, 8, 16, 0, 0),       # N = 128 exactly, no text
    (1, 1, 1, 0, 0, 0, 0),        # N = 1
    (1, 2, 5, 1, 1, 0, 0),        # N = 6
    (1, 2, 129, 0, 0, 0, 0),      # text only, N = 129
    (2, 2, 64, 16, 16, 3, 5),     # N = 335 with a reference stream
    (1, 3, 3, 11, 23, 0, 0),      # N = 256, two full tiles
    (1, 2, 0, 0, 0, 7, 9),        # reference only
    (1, 1, 100, 20, 20, 0, 0),    # N = 500
]


@pytest.mark.parametrize("B,H,txt,ih,iw,rh,rw", RAGGED)
def test_ragged_geometry_every_row(B, H, txt, ih, iw, rh, rw):
    w = synthetic.Workload("ragged", B, H, txt, ih, iw, rh, rw)
    inp = synthetic.make_inputs(w, seed=B * 1000 + txt)
    out, _ = _run(w, inp)
    want = oracle.attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k)
    compare(host_f64(out), want, BF16_MAX_ABS, BF16_MEAN_ABS, BF16_REL_RMS, "ragged %s" % (w.tokens,))


@pytest.mark.parametrize("name,per_head,full_head", [
    ("flux_1024_4608", 24, True),
    ("flux_2048_16896", 8, False),
    ("i2i_2048_33280", 4, False),
])
def test_full_size_sampled_rows(name, per_head, full_head):
    w = synthetic.WORKLOADS[name]
    inp = synthetic.make_inputs(w)
    n = w.tokens
    out, _ = _run(w, inp)
    got_all = out.float().cpu().numpy()
    assert np.all(np.isfinite(got_all))
    rows = synthetic.sample_rows(w, n, per_head)
    if full_head:
        extra = np.stack([np.zeros(n, np.int64), np.full(n, w.heads - 1, np.int64), np.arange(n)], 1)
        rows = np.concatenate([rows, extra], 0)
    want = oracle.attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k, rows=rows)
    got = gather_rows(got_all, rows).astype(np.float64)
    compare(got, want, BF16_MAX_ABS, BF16_MEAN_ABS, BF16_REL_RMS, name)


def test_inputs_are_not_modified():
    w = synthetic.WORKLOADS["tiny_320"]
    inp = synthetic.make_inputs(w)
    d = device_inputs(inp)
    before = [d[x].clone() for x in ("q", "k", "v")]
    attn = fa.FluxAttention(w.batch, w.heads, 320)
    attn.forward(d["q"], d["k"], d["v"], *_geom(w, 320), d["q_norm_w"], d["k_norm_w"])
    assert attn.sync_status() == 0
    for a, x in zip(before, ("q", "k", "v")):
        assert torch.equal(a, d[x])


def test_zero_tokens_is_a_no_op():
    attn = fa.FluxAttention(1, 2, 64)
    z = torch.empty((1, 0, 2, 128), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(128, device="cuda")
    out = attn.forward(z, z, z, 0, 0, 0, 0, 0, w, w, out=torch.empty_like(z))
    assert out.numel() == 0
    assert attn.sync_status() == 0


def test_invalid_arguments_are_rejected_on_the_host():
    w = synthetic.WORKLOADS["tiny_320"]
    inp = synthetic.make_inputs(w)
    d = device_inputs(inp)
    h = fa.flux_attn_create(1, 2, 320)
    args = lambda **kw: dict(dict(q=d["q"], k=d["k"], v=d["v"], out=torch.empty_like(d["q"]),
                                  wq=d["q_norm_w"], wk=d["k_norm_w"], geom=(64, 16, 16, 0, 0)), **kw)

    def call(a):
        fa.flux_attn_forward(h, a["q"], a["k"], a["v"], *a["geom"], None, a["wq"], a["wk"], a["out"])

    # a pointer 4 KB before the end of its own allocation: far too small for out
    from cuda.bindings import driver as cudrv
    from cuda.bindings import runtime as cudart
    err, raw = cudart.cudaMalloc(1 << 20)
    assert int(err) == 0
    err, base, size = cudrv.cuMemGetAddressRange(raw)
    assert int(err) == 0
    near_end = int(base) + int(size) - 4096
    host = torch.zeros(1, 320, 2, 128, dtype=torch.bfloat16)
    bad = [
        args(geom=(65, 16, 16, 0, 0)),                           # N > max_tokens
        args(geom=(-1, 16, 16, 0, 0)),                           # negative geometry
        args(q=host.data_ptr()),                                 # host memory
        args(out=near_end),                                      # too small
        args(v=d["v"].data_ptr() + 2),                           # misaligned
        args(wq=None),                                           # missing weight
        args(out=d["q"]),                                        # aliasing
    ]
    try:
        for a in bad:
            with pytest.raises(fa.FluxAttnError) as e:
                call(a)
            assert e.value.status == fa.FLUX_ATTN_ERR_INVALID_ARG, str(e.value)
    finally:
        cudart.cudaFree(raw)
    # the handle is still good afterwards
    out = torch.empty_like(d["q"])
    call(args(out=out))
    assert fa.flux_attn_sync_status(h) == 0
    fa.flux_attn_destroy(h)


def test_forced_device_timeout_is_reported_and_recoverable():
    w = synthetic.WORKLOADS["tiny_320"]
    inp = synthetic.make_inputs(w)
    d = device_inputs(inp)
    bad = fa.FluxAttention(1, 2, 320, debug_flags=fa.FLUX_ATTN_DEBUG_FORCE_TIMEOUT)
    bad.forward(d["q"], d["k"], d["v"], *_geom(w, 320), d["q_norm_w"], d["k_norm_w"])
    assert bad.sync_status() == fa.FLUX_ATTN_ERR_DEVICE_TIMEOUT
    assert bad.sync_status() == 0          # the word was cleared
    bad.close()
    out, _ = _run(w, inp)                  # the context is still usable
    want = oracle.attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k)
    compare(host_f64(out), want, BF16_MAX_ABS, BF16_MEAN_ABS, BF16_REL_RMS, "after timeout")
