"""The per-row bound of the FP8 attention's P rounding, checked on the CPU.

The GPU tests hold every FP8 output row to the bound of tests/fp8_bound.py.
Before that bound is trusted it is pinned here against an fp64 simulation of
the method ("Speed up image generation with FLUX 3 Image Klein on NVIDIA
Blackwell GPUs", section "Quantized and sparse attention": P.V in FP8): on the
oracle's dequantised Q', K', V, blocks of 128 keys, a running row max, P
stored as E4M3 of 256 p (round to nearest even), O and l rescaled when the max
moves, l the sum of the stored values.  The simulation must stay inside the
bound on every row of the edge shapes with 1 % x8 outliers; a simulation with
a plausible slip (P truncated to E4M3 instead of rounded, or P rounded to
two mantissa bits) must leave either the bound or the relative-RMS gate of the
GPU tests, which the simulation of the method itself keeps.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import fp8_bound as fb
from gpu_util import FP8_REL_RMS

SHAPES = [
    (2, 2, 64, 16, 16, 0, 0),     # the tiny case, N = 320
    (1, 2, 7, 5, 9, 0, 0),        # N = 52, one partial tile
    (1, 2, 129, 0, 0, 0, 0),      # text only, a second tile with one key
    (2, 2, 64, 16, 16, 3, 5),     # N = 335 with a reference stream
    (1, 2, 0, 0, 0, 7, 9),        # reference only
]


def _e4m3(x, mode):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if mode == "rne":
        return t.to(torch.float8_e4m3fn).to(torch.float64).numpy()
    if mode == "trunc":   # drop the mantissa bits below the third (toward zero)
        u = t.view(torch.int32) & ~((1 << 20) - 1)
        return u.view(torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    if mode == "two_bits":
        m, e = np.frexp(x)
        return np.ldexp(np.round(m * 8.0) / 8.0, e)
    raise ValueError(mode)


def simulate(qd, kd, vd, ns, mode="rne", bn=128):
    """The kernel's method in fp64: running max in log2 units, P = code of 256 p."""
    s = qd[ns] @ kd.T / np.sqrt(qd.shape[1]) / np.log(2.0)
    R, N = s.shape
    m = np.full(R, -np.inf)
    l = np.zeros(R)
    O = np.zeros((R, vd.shape[1]))
    for j0 in range(0, N, bn):
        sb = s[:, j0:j0 + bn]
        mn = np.maximum(m, sb.max(axis=1))
        alpha = np.where(np.isfinite(m), np.exp2(m - mn), 0.0)
        pt = _e4m3(256.0 * np.exp2(sb - mn[:, None]), mode)
        l = l * alpha + pt.sum(axis=1)
        O = O * alpha[:, None] + pt @ vd[j0:j0 + bn]
        m = mn
    return O / l[:, None]


def _run(shape, seed, mode):
    """(worst ratio to the bound, squared-error sum, squared-output sum) of the
    simulated method on every row of one edge shape."""
    B, H, txt, ih, iw, rh, rw = shape
    w = synthetic.Workload("fp8_bound", B, H, txt, ih, iw, rh, rw, precision="fp8", outliers=True)
    inp = synthetic.make_inputs(w, seed=seed)
    worst, se, so = 0.0, 0.0, 0.0
    for b in range(B):
        for h in range(H):
            qd, kd, vd = fb.dequantised_head(inp, b, h)
            ns = np.arange(w.tokens)
            o, p, l = fb.head_rows(qd, kd, vd, ns)
            bnd = fb.bound_from(o, p, l, vd)
            got = simulate(qd, kd, vd, ns, mode)
            worst = max(worst, float((np.abs(got - o) / bnd).max()))
            se += float(((got - o) ** 2).sum())
            so += float((o ** 2).sum())
    return worst, se, so


@pytest.mark.parametrize("shape", SHAPES)
def test_the_method_stays_inside_the_bound_and_the_rms_gate(shape):
    worst, se, so = _run(shape, seed=shape[2] + 7, mode="rne")
    assert worst <= 1.0
    assert np.sqrt(se / so) <= FP8_REL_RMS


@pytest.mark.parametrize("mode", ["trunc", "two_bits"])
def test_a_slip_in_the_p_rounding_is_caught(mode):
    """Truncated P, or P with two mantissa bits (the E5M2 format's), stays inside
    the worst-case bound -- a uniform relative bias cancels in o = sum p v / sum p
    -- but doubles the relative RMS error, which the gate of the GPU tests
    catches over these shapes."""
    runs = [_run(s, seed=s[2] + 7, mode=mode) for s in SHAPES]
    worst = max(r[0] for r in runs)
    rel_rms = np.sqrt(sum(r[1] for r in runs) / sum(r[2] for r in runs))
    assert worst > 1.0 or rel_rms > FP8_REL_RMS, (worst, rel_rms)


def test_helper_rows_equal_the_oracle():
    """fp8_bound's own fp64 attention over the dequantised inputs is the oracle's."""
    w = synthetic.Workload("fp8_bound", 1, 2, 9, 5, 7, precision="fp8", outliers=True)
    inp = synthetic.make_inputs(w, seed=3)
    rows = fb.all_rows(w)
    o, _ = fb.rows_and_bounds(inp, rows)
    want = oracle.attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k, rows=rows, fp8=True)
    np.testing.assert_allclose(o, want, rtol=0, atol=1e-12)
