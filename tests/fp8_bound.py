"""Per-row error bound of the FP8 attention's probability rounding (test helper).

"Speed up image generation with FLUX 3 Image Klein on NVIDIA Blackwell GPUs",
section "Quantized and sparse attention": P.V runs in FP8 (v_dtype fp8).  The
oracle attends exactly over its own dequantised Q', K', V and does not round
P; the GPU stores p (relative to the running row max, scaled by 256) as E4M3
codes p~ and divides sum p~ v~ by the sum of the same p~.  With
o = sum p v~ / sum p (the oracle) and p~_m = p_m + d_m,

    o_gpu - o = sum_m d_m (v~_m - o) / sum_m p~_m                  (sum p (v~ - o) = 0)

so, per output element i,

    |o_gpu,i - o_i| <= sum_m e_m |v~_mi - o_i| / (l - sum_m e_m)
                       + (2^-8 + 2^-9) |o_i| + 1e-5

with p in units where the row max is 1 (p_m = exp(s_m - s_max), l = sum p),
  e_m = 2^-4 p_m (1 + 2^-6)   the E4M3 half step (three mantissa bits), widened
                              by 2^-6 for the fp32 score and exp2 arithmetic
        + 2^-18               the subnormal E4M3 step (2^-10 of a code of 256)
                              when 256 p < 2^-6, in the same units,
  2^-8 |o_i|                  the row sum: exact in fp32 for the E4M3 blocks
                              (P times ones on the tensor core); the BF16
                              repair blocks of the VC instance weight V by
                              bf16(p) but add the unrounded p, a mismatch of
                              at most 2^-9 |o_i|,
  2^-9 |o_i|                  the bf16 rounding of the output.

Everything here is computed in fp64 from the oracle's dequantised inputs
(oracle.fp8_quantize_head), never from the GPU's.
"""
from __future__ import annotations

import numpy as np

import oracle

E4M3_HALF_STEP = 2.0 ** -4
SUBNORMAL_STEP = 2.0 ** -18
ROW_SUM_REL = 2.0 ** -8
BF16_OUT_REL = 2.0 ** -9
ABS_FLOOR = 1e-5

_DECODE = None


def _decode_table():
    global _DECODE
    if _DECODE is None:
        _DECODE = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    return _DECODE


def dequantised_head(inp, b: int, h: int):
    """The oracle's dequantised Q', K', V of head (b, h): float64 [N, 128] each."""
    q8, k8, v8, sc = oracle.fp8_quantize_head(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k, b, h)
    t = _decode_table()
    return t[q8] * sc[0], t[k8] * sc[1], t[v8] * sc[2]


def head_rows(qd, kd, vd, ns):
    """Exact attention rows ns of one head over dequantised inputs, with the
    bound terms: returns (o, p, l) with p [R, N] in units of the row max."""
    s = qd[ns] @ kd.T / np.sqrt(qd.shape[1])
    p = np.exp(s - s.max(axis=1, keepdims=True))
    l = p.sum(axis=1, keepdims=True)
    o = p @ vd / l
    return o, p, l


def bound_from(o, p, l, vd):
    """Per-element bound [R, d] of the P-rounding error (module docstring)."""
    e = E4M3_HALF_STEP * (1.0 + 2.0 ** -6) * p + SUBNORMAL_STEP
    if p.shape[0] * p.shape[1] * vd.shape[1] <= 1 << 24:
        num = np.einsum("rm,rmi->ri", e, np.abs(vd[None, :, :] - o[:, None, :]))
    else:
        num = np.stack([e[r] @ np.abs(vd - o[r]) for r in range(p.shape[0])])
    den = l[:, 0] - e.sum(axis=1)
    return num / den[:, None] + (ROW_SUM_REL + BF16_OUT_REL) * np.abs(o) + ABS_FLOOR


def rows_and_bounds(inp, rows):
    """o and its bound for (b, h, n) rows (int64 [R, 3]), in the order given."""
    d = inp.q.shape[-1]
    o = np.empty((len(rows), d))
    bnd = np.empty((len(rows), d))
    heads = {}
    for i, (b, h, _) in enumerate(rows):
        heads.setdefault((int(b), int(h)), []).append(i)
    for (b, h), idx in heads.items():
        qd, kd, vd = dequantised_head(inp, b, h)
        ns = rows[idx, 2]
        ob, p, l = head_rows(qd, kd, vd, ns)
        o[idx] = ob
        bnd[idx] = bound_from(ob, p, l, vd)
    return o, bnd


def all_rows(w):
    bb, hh, nn = np.meshgrid(np.arange(w.batch), np.arange(w.heads), np.arange(w.tokens), indexing="ij")
    return np.stack([bb.ravel(), hh.ravel(), nn.ravel()], 1).astype(np.int64)


def check_rows(got, want, bound, what=""):
    """Every element of every row within its bound; returns the worst ratio."""
    assert got.shape == want.shape == bound.shape, (got.shape, want.shape, bound.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite output" % what
    ratio = np.abs(got - want) / bound
    worst = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
    assert ratio.max() <= 1.0, "%s: row %d elem %d off by %.3e, bound %.3e (ratio %.2f)" % (
        what, worst[0], worst[1], abs(got[worst] - want[worst]), bound[worst], ratio.max())
    return float(ratio.max())


# ------------------------------------------------------- VC-Attention repair

def vc_dequantised_head(inp, b: int, h: int, rho: float):
    """The oracle's inputs of VC-Attention for head (b, h) (reading R7 of the
    oracle): dequantised Q', and K', V dequantised except the repaired tokens,
    which keep their exact values.  Returns (q, k, v, repaired token indices)."""
    qd, kd, vd = dequantised_head(inp, b, h)
    sel, _ = oracle.vc_select_head(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k, rho, b, h)
    kx = oracle.prologue(np.ascontiguousarray(inp.k[b:b + 1, :, h:h + 1, :]), inp.pos, inp.w_k)[0, :, 0, :]
    vx = (inp.v[b, :, h, :].astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    kd[sel] = kx[sel]
    vd[sel] = vx[sel]
    return qd, kd, vd, sel


def vc_rows_and_bounds(inp, rows, rho: float):
    """o and its bound for (b, h, n) rows of VC-Attention.  On top of the P
    rounding bound, a repaired key carries the GPU's bf16 copies of k' / s_k and
    v / s_v (relative half step 2^-9): its score moves by at most
    2^-9 sum_d |q_d k_d| / sqrt(d) (a relative change of p of about as much)
    and its value by 2^-9 |v|."""
    d = inp.q.shape[-1]
    o = np.empty((len(rows), d))
    bnd = np.empty((len(rows), d))
    heads = {}
    for i, (b, h, _) in enumerate(rows):
        heads.setdefault((int(b), int(h)), []).append(i)
    for (b, h), idx in heads.items():
        qd, kd, vd, sel = vc_dequantised_head(inp, b, h, rho)
        ns = rows[idx, 2]
        ob, p, l = head_rows(qd, kd, vd, ns)
        bb = bound_from(ob, p, l, vd)
        ds = 2.0 ** -9 * (np.abs(qd[ns]) @ np.abs(kd[sel]).T) / np.sqrt(d)     # [R_rows, R_sel]
        ps = p[:, sel] * 1.01 * np.expm1(ds)                                   # p change of a repaired key
        bb += (ps[:, :, None] * np.abs(vd[sel][None, :, :] - ob[:, None, :])).sum(axis=1) / l
        bb += 2.0 ** -9 * (p[:, sel] @ np.abs(vd[sel])) / l
        o[idx] = ob
        bnd[idx] = bb
    return o, bnd
