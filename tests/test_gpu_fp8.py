"""FP8 (E4M3) joint attention through the C ABI against the fp64 oracle (GPU).

The oracle quantises its own fp64 Q', K', V per (batch, head) with
scale = amax / 448 and attends exactly over the dequantised values.  The GPU
also stores P as E4M3 codes of 256 p, which the oracle does not: every output
element of every checked row must lie within the bound that rounding allows
(tests/fp8_bound.py, pinned against an fp64 simulation of the method in
tests/test_fp8_bound.py), and the relative RMS error of each case within the
gate of tests/gpu_util.py.  The FP8 classifier-free-guidance pair at 2048^2
(N = 16896) must also meet max-abs 6e-2.  The prologue's E4M3 codes are
compared code by code: the GPU computes Q', K' in fp32, so a value that sits
within fp32 rounding of a midpoint between two codes may land on the
neighbouring code, and nothing else may differ.

Inputs: the FP8 workload's N(0, 1) values with 1 % outliers at x8 in every
case, including the edge shapes (N <= 335) where one x8 outlier row of V can
carry a tenth of a row's weight; there the rounding of P alone moves an output
by up to 0.17 (the simulation), which the per-row bound accounts for.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import FP8_MAX_ABS, FP8_REL_RMS, compare, device_inputs, gather_rows, host_f64, v8t_token_order
import fp8_bound as fb

pytestmark = pytest.mark.gpu

import diffusion_transformer_joint_txt_b300 as fa  # noqa: E402

DECODE = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))


def _fp8(name, B, H, txt, ih, iw, rh=0, rw=0, outliers=True):
    return synthetic.Workload(name, B, H, txt, ih, iw, rh, rw, precision="fp8", outliers=outliers)


def _geom(w):
    return w.txt_len, w.img_h, w.img_w, w.ref_h, w.ref_w


def _forward(w, inp, handle=None):
    d = device_inputs(inp)
    attn = handle or fa.FluxAttention(w.batch, w.heads, w.tokens, precision="fp8")
    out = attn.forward(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    assert attn.sync_status() == 0
    return out, attn


def _check_rows(out, inp, w, rows=None, max_abs=None, what=""):
    """Every element of the given rows (all rows when None) within its P-rounding
    bound, the case's relative RMS error within the gate, and max-abs when given."""
    got_all = out.float().cpu().numpy().astype(np.float64)
    rows = fb.all_rows(w) if rows is None else rows
    got = gather_rows(got_all, rows)
    want, bound = fb.rows_and_bounds(inp, rows)
    oracle_rows = oracle.attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k, rows=rows, fp8=True)
    np.testing.assert_allclose(want, oracle_rows, rtol=0, atol=1e-10)
    fb.check_rows(got, want, bound, what=what)
    compare(got, want, max_abs if max_abs is not None else np.inf, rel_rms=FP8_REL_RMS, what=what)


def _codes_match(got: np.ndarray, want: np.ndarray, what: str):
    """Equal codes, except rare neighbours (one E4M3 step apart)."""
    assert got.shape == want.shape, (got.shape, want.shape)
    diff = got != want
    frac = float(diff.mean())
    assert frac <= 1e-4, "%s: %.2e of the codes differ" % (what, frac)
    if diff.any():
        a, b = DECODE[got[diff]], DECODE[want[diff]]
        step = np.maximum(np.abs(b), 2.0 ** -6) * 2.0 ** -3   # one mantissa step (subnormal floor)
        assert np.all(np.abs(a - b) <= step * 1.0001), what


@pytest.mark.parametrize("B,H,txt,ih,iw,rh,rw", [
    (2, 3, 7, 5, 9, 2, 3),        # N = 58, Npad = 64: fewer tokens than warps of the grid
    (2, 3, 80, 30, 40, 20, 36),   # N = 2000: every warp's tokens span both batch rows
    (1, 40, 60, 20, 32, 0, 0),    # N = 700, H = 40: four warps per block instead of eight
])
def test_fp8_prologue_codes_and_scales(B, H, txt, ih, iw, rh, rw):
    w = _fp8("fp8_prologue", B, H, txt, ih, iw, rh, rw)
    inp = synthetic.make_inputs(w, seed=3)
    d = device_inputs(inp)
    n = w.tokens
    attn = fa.FluxAttention(w.batch, w.heads, n, precision="fp8")
    q8, k8, v8t, scales = attn.prologue_fp8(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    assert attn.sync_status() == 0
    q8, k8, v8t, scales = (t.cpu().numpy() for t in (q8, k8, v8t, scales))
    assert v8t.shape[-1] == fa.pad16(n)
    v8t = v8t_token_order(v8t)
    for b in range(w.batch):
        for h in range(w.heads):
            oq, ok, ov, osc = oracle.fp8_quantize_head(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k, b, h)
            np.testing.assert_allclose(scales[b, h].astype(np.float64), osc, rtol=1e-5)
            _codes_match(q8[b, h], oq, "q8 (%d, %d)" % (b, h))
            _codes_match(k8[b, h], ok, "k8 (%d, %d)" % (b, h))
            # V is bf16 and its amax a bf16 value: (448 x) / amax rounds once, so
            # every code equals the oracle's (the case N = 700, H = 40 holds
            # exact midpoints between codes: amax 24.5 makes x / scale = 128 x / 7)
            np.testing.assert_array_equal(v8t[b, h, :, :n], ov.T, "v8t (%d, %d)" % (b, h))
            assert not v8t[b, h, :, n:].any(), "padding columns of V^T are not zero"


def test_fp8_v_codes_exact_on_adversarial_heads():
    """V^T codes equal the oracle's code for code on heads built to break a
    quotient that is not rounded once: bf16 values with amax 24.5 (many
    x / scale = 128 x / 7 exactly halfway between two codes, where a product
    with a rounded 448 / amax takes the odd code) and with amax 30.5 (ties
    that a scale rounded first misses), amax 2^65 with tiny negative values
    (2^-E x underflows; the code of -0 must survive), an all-zero head
    (scale 1) and a head of subnormal bf16 values."""
    w = _fp8("fp8_vcodes", 1, 5, 40, 10, 26, 0, 0)          # N = 300
    inp = synthetic.make_inputs(w, seed=5)
    rng = np.random.default_rng(11)
    n = w.tokens
    heads = np.zeros((5, n, 128), np.float32)
    heads[0] = rng.uniform(-24.5, 24.5, (n, 128))
    heads[0, 17, 3] = 24.5
    heads[0, 5, :8] = 203.0 / 4096 * np.array([1, -1, 2, -2, 4, -4, 8, -8])   # exact ties
    heads[1] = rng.standard_normal((n, 128)) * 2.0 ** -130
    heads[1, 0, 0] = 2.0 ** 65
    heads[3] = rng.standard_normal((n, 128)) * 2.0 ** -128
    heads[4] = rng.uniform(-30.5, 30.5, (n, 128))
    heads[4, 17, 3] = 30.5
    heads[4, 5, :8] = 183.0 / 2048 * np.array([1, -1, 2, -2, 4, -4, 8, -8])   # exact ties
    inp.v[0] = synthetic.bf16_bits_from_f32(heads.transpose(1, 0, 2))
    d = device_inputs(inp)
    attn = fa.FluxAttention(w.batch, w.heads, n, precision="fp8")
    _, _, v8t, scales = attn.prologue_fp8(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    assert attn.sync_status() == 0
    v8t, scales = v8t_token_order(v8t.cpu().numpy()), scales.cpu().numpy()
    for h in range(5):
        _, _, ov, osc = oracle.fp8_quantize_head(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k, 0, h)
        assert scales[0, h, 2] == np.float32(osc[2]), h
        np.testing.assert_array_equal(v8t[0, h, :, :n], ov.T, "head %d" % h)
    assert np.any(v8t[0, 1, :, :n] == 0x80)          # the code of -0 is there


def test_fp8_tiny_every_row():
    w = _fp8("fp8_tiny", 2, 2, 64, 16, 16)
    inp = synthetic.make_inputs(w)
    out, _ = _forward(w, inp)
    _check_rows(out, inp, w, what="fp8 tiny")


RAGGED = [
    (1, 2, 7, 5, 9, 0, 0),        # N = 52, one partial tile, Npad = 64
    (1, 1, 1, 0, 0, 0, 0),        # N = 1
    (1, 2, 129, 0, 0, 0, 0),      # text only, N = 129: a second tile with one key
    (2, 2, 64, 16, 16, 3, 5),     # N = 335 with a reference stream
    (1, 2, 0, 0, 0, 7, 9),        # reference only
    (1, 3, 3, 11, 23, 0, 0),      # N = 256, two full tiles
]


@pytest.mark.parametrize("B,H,txt,ih,iw,rh,rw", RAGGED)
def test_fp8_ragged_every_row(B, H, txt, ih, iw, rh, rw):
    w = _fp8("fp8_ragged", B, H, txt, ih, iw, rh, rw)
    inp = synthetic.make_inputs(w, seed=B * 100 + txt)
    out, _ = _forward(w, inp)
    _check_rows(out, inp, w, what="fp8 ragged N=%d" % w.tokens)


def test_fp8_cfg_pair_full_size_sampled_rows():
    """32 random query rows of every (b, h) plus the boundary rows (first and
    last text and image tokens, tile edges, row N - 1)."""
    w = synthetic.WORKLOADS["fp8_cfg_2048_16896"]
    inp = synthetic.make_inputs(w)
    out, _ = _forward(w, inp)
    assert bool(torch.isfinite(out.float()).all())
    rows = synthetic.sample_rows(w, w.tokens, 32)
    _check_rows(out, inp, w, rows=rows, max_abs=FP8_MAX_ABS, what=w.name)


def test_fp8_split_calls_equal_forward_and_are_deterministic():
    w = _fp8("fp8_split", 1, 2, 64, 16, 16)
    inp = synthetic.make_inputs(w, seed=4)
    d = device_inputs(inp)
    attn = fa.FluxAttention(w.batch, w.heads, w.tokens, precision="fp8")
    full = attn.forward(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    codes = attn.prologue_fp8(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    split = attn.attend_fp8(*codes)
    again = attn.forward(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    assert attn.sync_status() == 0
    assert torch.equal(full, split)
    assert torch.equal(full, again)


def test_fp8_all_zero_head_uses_unit_scale():
    w = _fp8("fp8_zero", 1, 2, 9, 4, 5)
    inp = synthetic.make_inputs(w, seed=6)
    for t in (inp.q, inp.k, inp.v):
        t[:, :, 1, :] = 0                                 # head 1 is all zero
    d = device_inputs(inp)
    attn = fa.FluxAttention(w.batch, w.heads, w.tokens, precision="fp8")
    q8, k8, v8t, scales = attn.prologue_fp8(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    out = attn.attend_fp8(q8, k8, v8t, scales)
    assert attn.sync_status() == 0
    assert torch.equal(scales[0, 1].cpu(), torch.ones(3))
    assert not out[:, :, 1, :].float().abs().max().item()
    rows = fb.all_rows(w)
    live = rows[rows[:, 1] == 0]                          # head 1 is exactly zero (checked above)
    _check_rows(out, inp, w, rows=live, what="fp8 zero head")


def test_fp8_handle_rejects_bf16_steps_and_vice_versa():
    w = _fp8("fp8_mix", 1, 2, 8, 2, 4)
    inp = synthetic.make_inputs(w)
    d = device_inputs(inp)
    f8 = fa.FluxAttention(1, 2, w.tokens, precision="fp8")
    with pytest.raises(fa.FluxAttnError) as e:
        f8.prologue(d["q"], d["k"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    assert e.value.status == fa.FLUX_ATTN_ERR_INVALID_ARG
    bf = fa.FluxAttention(1, 2, w.tokens)
    with pytest.raises(fa.FluxAttnError) as e:
        bf.prologue_fp8(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    assert e.value.status == fa.FLUX_ATTN_ERR_INVALID_ARG


def test_fp8_forced_device_timeout_is_reported():
    w = _fp8("fp8_timeout", 1, 2, 64, 16, 16)
    inp = synthetic.make_inputs(w)
    d = device_inputs(inp)
    bad = fa.FluxAttention(1, 2, w.tokens, precision="fp8", debug_flags=fa.FLUX_ATTN_DEBUG_FORCE_TIMEOUT)
    bad.forward(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    assert bad.sync_status() == fa.FLUX_ATTN_ERR_DEVICE_TIMEOUT
    bad.close()
    out, _ = _forward(w, inp)
    _check_rows(out, inp, w, what="fp8 after timeout")
