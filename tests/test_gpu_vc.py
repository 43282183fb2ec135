"""VC-Attention FP8 through the C ABI against the fp64 oracle (GPU).

"Speed up image generation with FLUX 3 Image Klein on NVIDIA Blackwell GPUs",
section "Quantized and sparse attention": VC-Attention FP8 with a repair
budget -- the worst-quantised share of the tokens gets its quantisation
residual corrected (reading R7 of the oracle: per (b, h) the ceil(rho N) key
tokens of largest |k' - deq(k')|^2 + |v - deq(v)|^2 attend with their exact
K', V).

What is compared:
  * the repair set (index work): the GPU's set equals the oracle's, except
    where the two errors that decide it lie within 1e-5 (relative) of each
    other -- the GPU takes the decision on its fp32 K', the oracle on fp64;
  * the moved codes: the first N - R key positions hold exactly the plain
    FP8 prologue's codes of the non-repaired tokens, in the documented order;
  * the repaired rows: k_rep s_k and v_rep s_v within bf16 rounding of the
    oracle's exact K' and V;
  * the output: every element of every checked row within the P-rounding
    bound of tests/fp8_bound.py (with the repaired keys' bf16 terms), the
    relative RMS error within the FP8 gate, and max-abs 6e-2 on the CFG pair
    at 2048^2 with the page's budget 0.005.
Inputs: the FP8 workload's N(0, 1) draws with 1 % outliers at x8.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import fp8_bound as fb
from gpu_util import FP8_MAX_ABS, FP8_REL_RMS, compare, device_inputs, gather_rows, v8t_token_order

pytestmark = pytest.mark.gpu

import diffusion_transformer_joint_txt_b300 as fa  # noqa: E402

PAGE_BUDGET = 0.005


def _f32(rho):
    """The budget as the library holds it (a float in the config): the oracle
    gets the same value, so that both take R = ceil(rho N) of one number."""
    return float(np.float32(rho))


def _fp8(name, B, H, txt, ih, iw, rh=0, rw=0):
    return synthetic.Workload(name, B, H, txt, ih, iw, rh, rw, precision="fp8", outliers=True)


def _geom(w):
    return w.txt_len, w.img_h, w.img_w, w.ref_h, w.ref_w


def _check_selection(idx, inp, w, rho):
    """GPU repair sets (int32 [B, H, R]) against the oracle's, near-ties allowed."""
    R = oracle.vc_repair_count(rho, w.tokens)
    assert idx.shape[-1] == R
    for b in range(w.batch):
        for h in range(w.heads):
            got = idx[b, h].astype(np.int64)
            assert np.all(np.diff(got) > 0) and got.min() >= 0 and got.max() < w.tokens, (b, h)
            want, err = oracle.vc_select_head(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k, rho, b, h)
            if np.array_equal(got, want):
                continue
            e_r = np.sort(err)[::-1][R - 1]                       # the deciding error
            for m in np.setdiff1d(got, want):
                assert err[m] >= e_r * (1 - 1e-5), ("head", b, h, "token", m, err[m], e_r)
            for m in np.setdiff1d(want, got):
                assert err[m] <= e_r * (1 + 1e-5), ("head", b, h, "token", m, err[m], e_r)


def _check_output(out, inp, w, rho, rows=None, max_abs=None, what=""):
    rows = fb.all_rows(w) if rows is None else rows
    got = gather_rows(out.float().cpu().numpy().astype(np.float64), rows)
    want, bound = fb.vc_rows_and_bounds(inp, rows, rho)
    np.testing.assert_allclose(want, oracle.vc_attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k, rho,
                                                              rows=rows), rtol=0, atol=1e-10)
    fb.check_rows(got, want, bound, what=what)
    compare(got, want, max_abs if max_abs is not None else np.inf, rel_rms=FP8_REL_RMS, what=what)


CASES = [
    # B, H, txt, img_h, img_w, ref_h, ref_w, rho
    (2, 2, 64, 16, 16, 0, 0, PAGE_BUDGET),   # N = 320, R = 2: one repair block, most keys E4M3
    (1, 3, 7, 5, 9, 0, 0, 0.1),              # N = 52, R = 6, one partial E4M3 block
    (1, 2, 60, 20, 32, 0, 0, 0.3),           # N = 700, R = 210: two repair blocks
    (2, 2, 64, 16, 16, 3, 5, 0.05),          # N = 335 with a reference stream, B = 2
    (1, 2, 5, 10, 12, 0, 0, 1.0),            # N = 125, every key repaired: no E4M3 key block
    (1, 2, 129, 0, 0, 0, 0, 127.5 / 129),    # R = 128 of 129: one E4M3 key left
]


@pytest.mark.parametrize("B,H,txt,ih,iw,rh,rw,rho", CASES)
def test_vc_every_row_and_every_step(B, H, txt, ih, iw, rh, rw, rho):
    rho = _f32(rho)
    w = _fp8("vc", B, H, txt, ih, iw, rh, rw)
    inp = synthetic.make_inputs(w, seed=B * 31 + txt)
    d = device_inputs(inp)
    n = w.tokens
    attn = fa.FluxAttention(B, H, n, precision="fp8", vc_repair_budget=rho)
    R = attn.vc_repair_count(n)
    assert R == oracle.vc_repair_count(rho, n) and R > 0
    q8, k8, v8t, scales, idx, k_rep, v_rep = attn.prologue_fp8_vc(d["q"], d["k"], d["v"], *_geom(w),
                                                                  d["q_norm_w"], d["k_norm_w"])
    out = attn.attend_fp8_vc(q8, k8, v8t, scales, k_rep, v_rep)
    full = attn.forward(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    assert attn.sync_status() == 0
    assert torch.equal(out, full)
    idx_h = idx.cpu().numpy()
    _check_selection(idx_h, inp, w, rho)
    # codes: the plain FP8 prologue's, with the repaired tokens moved out of [0, N - R)
    plain = fa.FluxAttention(B, H, n, precision="fp8")
    pq8, pk8, pv8t, psc = plain.prologue_fp8(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    assert plain.sync_status() == 0
    assert torch.equal(q8, pq8) and torch.equal(scales, psc)
    k8h, v8h, pk8h, pv8h = (t.cpu().numpy() for t in (k8, v8t, pk8, pv8t))
    # both prologues store V^T in the attention's key order: back to positions
    v8h, pv8h = v8t_token_order(v8h), v8t_token_order(pv8h)
    split = n - R
    for b in range(B):
        for h in range(H):
            chosen = set(idx_h[b, h].tolist())
            holes = [m for m in sorted(chosen) if m < split]
            fillers = [m for m in range(split, n) if m not in chosen]
            order = np.arange(split)
            order[holes] = fillers
            assert len(set(order.tolist()) & chosen) == 0
            np.testing.assert_array_equal(k8h[b, h, :split], pk8h[b, h, order], "k8 (%d, %d)" % (b, h))
            np.testing.assert_array_equal(v8h[b, h, :, :split], pv8h[b, h, :, order].T, "v8t (%d, %d)" % (b, h))
            # the repaired rows, in repair-set order, in the units of the codes
            sel = idx_h[b, h]
            kx = oracle.prologue(np.ascontiguousarray(inp.k[b:b + 1, :, h:h + 1, :]), inp.pos, inp.w_k)[0, :, 0, :]
            vx = synthetic.bf16_bits_to_f32(inp.v[b, :, h, :]).astype(np.float64)
            s = scales[b, h].cpu().numpy().astype(np.float64)
            kr = k_rep[b, h].float().cpu().numpy().astype(np.float64) * s[1]
            vr = v_rep[b, h].float().cpu().numpy().astype(np.float64) * s[2]
            # bf16 rounding (2^-9 relative) of the fp32 K', whose own rounding is
            # relative to the O(1) terms of the norm and rotation (absolute 2^-16)
            np.testing.assert_allclose(kr, kx[sel], rtol=2 ** -8, atol=2 ** -16)
            np.testing.assert_allclose(vr, vx[sel], rtol=2 ** -8, atol=1e-30)
    _check_output(full, inp, w, rho, what="vc rho=%g N=%d" % (rho, n))


def test_vc_cfg_pair_full_size_page_budget():
    """The CFG pair at 2048^2 (B = 2, N = 16896) with the page's budget 0.005
    (R = 85 per head): selection of every head, then 32 random rows per head
    plus the boundary rows."""
    w = synthetic.WORKLOADS["fp8_cfg_2048_16896"]
    inp = synthetic.make_inputs(w)
    d = device_inputs(inp)
    attn = fa.FluxAttention(w.batch, w.heads, w.tokens, precision="fp8", vc_repair_budget=PAGE_BUDGET)
    assert attn.vc_repair_count(w.tokens) == 85
    q8, k8, v8t, scales, idx, k_rep, v_rep = attn.prologue_fp8_vc(d["q"], d["k"], d["v"], *_geom(w),
                                                                  d["q_norm_w"], d["k_norm_w"])
    out = attn.attend_fp8_vc(q8, k8, v8t, scales, k_rep, v_rep)
    assert attn.sync_status() == 0
    assert bool(torch.isfinite(out.float()).all())
    _check_selection(idx.cpu().numpy(), inp, w, _f32(PAGE_BUDGET))
    rows = synthetic.sample_rows(w, w.tokens, 32)
    _check_output(out, inp, w, _f32(PAGE_BUDGET), rows=rows, max_abs=FP8_MAX_ABS, what="vc " + w.name)


def test_vc_repairs_a_planted_token_and_helps_its_queries():
    """A key token planted as its head's worst-quantised one (V row at +-7 with
    the head's amax 7.75: 11.4 code steps of error per element) is repaired, and
    the repaired output is closer to the unquantised attention than plain FP8."""
    w = _fp8("vc_plant", 1, 2, 40, 8, 10)
    inp = synthetic.make_inputs(w, seed=41)
    rng = np.random.default_rng(41)
    row = np.where(rng.random(128) < 0.5, -7.0, 7.0).astype(np.float32)
    inp.v[0, 50, 1] = synthetic.bf16_bits_from_f32(row)
    other = synthetic.bf16_bits_to_f32(inp.v[0, 49, 1]).copy()
    other[0] = 7.75
    inp.v[0, 49, 1] = synthetic.bf16_bits_from_f32(other)
    d = device_inputs(inp)
    rho = 1.5 / w.tokens                                     # R = 2
    attn = fa.FluxAttention(1, 2, w.tokens, precision="fp8", vc_repair_budget=rho)
    _, _, _, _, idx, _, _ = attn.prologue_fp8_vc(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    out = attn.forward(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    plain_attn = fa.FluxAttention(1, 2, w.tokens, precision="fp8")
    plain = plain_attn.forward(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    assert attn.sync_status() == 0 and plain_attn.sync_status() == 0
    assert 50 in idx[0, 1].cpu().tolist()
    exact = oracle.attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k)[0, :, 1]
    err_vc = np.abs(out[0, :, 1].float().cpu().numpy() - exact).mean()
    err_fp8 = np.abs(plain[0, :, 1].float().cpu().numpy() - exact).mean()
    assert err_vc < err_fp8, (err_vc, err_fp8)


def test_vc_handle_rules():
    w = _fp8("vc_rules", 1, 2, 8, 2, 4)
    inp = synthetic.make_inputs(w)
    d = device_inputs(inp)
    vc = fa.FluxAttention(1, 2, w.tokens, precision="fp8", vc_repair_budget=0.2)
    with pytest.raises(fa.FluxAttnError) as e:                 # the plain FP8 steps refuse a VC handle
        vc.prologue_fp8(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    assert e.value.status == fa.FLUX_ATTN_ERR_INVALID_ARG
    for kw in (dict(precision="bf16", vc_repair_budget=0.1), dict(precision="fp8", vc_repair_budget=1.5),
               dict(precision="fp8", vc_repair_budget=-0.1)):
        with pytest.raises(fa.FluxAttnError) as e:
            fa.FluxAttention(1, 2, w.tokens, **kw)
        assert e.value.status == fa.FLUX_ATTN_ERR_INVALID_ARG
    assert fa.FluxAttention(1, 2, w.tokens, precision="fp8").vc_repair_count(w.tokens) == 0
    assert vc.launches_per_forward(w.tokens) == 7
