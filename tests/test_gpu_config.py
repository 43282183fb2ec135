"""Non-default RoPE / RMSNorm configurations through the C ABI against the
fp64 oracle (GPU): other axis splits, theta and eps reach every kernel that
rotates or normalises (prologue, FP8 quantiser, QKV epilogue)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import (BF16_MAX_ABS, BF16_MEAN_ABS, BF16_REL_RMS, FP8_MAX_ABS, FP8_REL_RMS, compare, dev_bf16,
                      device_inputs, host_f64)

pytestmark = pytest.mark.gpu

import diffusion_transformer_joint_txt_b300 as fa  # noqa: E402

CONFIGS = [
    dict(axes=(32, 48, 48), theta=1000.0, eps=1e-5),
    dict(axes=(8, 64, 56), theta=20000.0, eps=1e-6),
    dict(axes=(0, 64, 64), theta=10000.0, eps=1e-3),   # no first axis: text tokens unrotated
]


def _kw(c):
    return dict(axes_dim=c["axes"], rope_theta=c["theta"], rms_eps=c["eps"])


def _geom(w):
    return w.txt_len, w.img_h, w.img_w, w.ref_h, w.ref_w


@pytest.mark.parametrize("cfg", CONFIGS, ids=lambda c: "axes%s" % "-".join(map(str, c["axes"])))
def test_forward_with_other_rope_and_norm(cfg):
    w = synthetic.Workload("cfg", 2, 3, 40, 9, 11, 3, 4)    # 151 tokens, reference stream, positions up to 10
    inp = synthetic.make_inputs(w, seed=31)
    d = device_inputs(inp)
    attn = fa.FluxAttention(w.batch, w.heads, w.tokens, **_kw(cfg))
    out = attn.forward(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    qn, kn = attn.prologue(d["q"], d["k"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    assert attn.sync_status() == 0
    kw = dict(eps=cfg["eps"], theta=cfg["theta"], axes=cfg["axes"])
    want = oracle.attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k, **kw)
    compare(host_f64(out), want, BF16_MAX_ABS, BF16_MEAN_ABS, BF16_REL_RMS, "forward %s" % (cfg,))
    wq = oracle.prologue(inp.q, inp.pos, inp.w_q, **kw).transpose(0, 2, 1, 3)
    err = np.abs(host_f64(qn) - wq)
    assert np.all(err <= 2.0 ** -8 * np.abs(wq) + 1e-5), float(err.max())


@pytest.mark.parametrize("cfg", CONFIGS[:2], ids=lambda c: "axes%s" % "-".join(map(str, c["axes"])))
def test_fp8_with_other_rope_and_norm(cfg):
    w = synthetic.Workload("cfg8", 1, 2, 40, 9, 11, precision="fp8")
    inp = synthetic.make_inputs(w, seed=32)
    d = device_inputs(inp)
    attn = fa.FluxAttention(w.batch, w.heads, w.tokens, precision="fp8", **_kw(cfg))
    out = attn.forward(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    assert attn.sync_status() == 0
    want = oracle.attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k, fp8=True, eps=cfg["eps"],
                                 theta=cfg["theta"], axes=cfg["axes"])
    compare(host_f64(out), want, FP8_MAX_ABS, rel_rms=FP8_REL_RMS, what="fp8 %s" % (cfg,))


def test_qkv_with_other_rope_and_norm():
    cfg = CONFIGS[0]
    w = synthetic.Workload("cfgqkv", 1, 2, 20, 6, 7)
    inp = synthetic.make_qkv_inputs(w, 128, seed=33)
    attn = fa.FluxAttention(w.batch, w.heads, w.tokens, **_kw(cfg))
    qn, kn, v = attn.qkv(dev_bf16(inp.x), dev_bf16(inp.w), torch.from_numpy(inp.bias).cuda(), *_geom(w),
                         q_norm_w=torch.from_numpy(inp.w_q).cuda(), k_norm_w=torch.from_numpy(inp.w_k).cuda())
    assert attn.sync_status() == 0
    oq, ok, _ = oracle.qkv_rows(inp.x, inp.w, inp.bias, w.tokens, inp.pos, inp.w_q, inp.w_k, w.heads,
                                eps=cfg["eps"], theta=cfg["theta"], axes=cfg["axes"])
    for got, want in ((qn, oq), (kn, ok)):
        g = host_f64(got)[0].transpose(1, 0, 2)            # [N, H, 128]
        err = np.abs(g - want)
        assert np.all(err <= 2.0 ** -8 * np.abs(want) + 1e-5), float(err.max())


@pytest.mark.parametrize("precision", ["bf16", "fp8"])
def test_max_head_count(precision):
    """192 heads, the most a handle accepts: the prologue's stream kernel then
    runs one warp per block (whole tokens) and the FP8 passes one or two (half
    tokens of 96 heads); every output row against the oracle."""
    w = synthetic.Workload("maxh", 1, 192, 40, 8, 8, 0, 0, precision=precision, outliers=False)   # N = 104
    inp = synthetic.make_inputs(w, seed=41)
    d = device_inputs(inp)
    attn = fa.FluxAttention(w.batch, w.heads, w.tokens, precision=precision)
    out = attn.forward(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    assert attn.sync_status() == 0
    want = oracle.attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k, fp8=(precision == "fp8"))
    if precision == "fp8":
        compare(host_f64(out), want, FP8_MAX_ABS, rel_rms=FP8_REL_RMS, what="fp8, 192 heads")
    else:
        compare(host_f64(out), want, BF16_MAX_ABS, BF16_MEAN_ABS, BF16_REL_RMS, "bf16, 192 heads")
