"""Shared helpers of the GPU tests: move seeded inputs to the device, compare
against the oracle with the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances: BF16 max-abs 1e-2 and mean-abs 1e-3, FP8 max-abs 6e-2 (against
# the oracle on its own dequantised inputs) on the configurations those
# figures are stated for; plus an internal gate on the relative RMS error so
# that a small systematic error cannot hide under a loose absolute bound.
# FP8 output rows are also held, element by element, to the bound the E4M3
# rounding of P allows (tests/fp8_bound.py).  The FP8 gate sits above the noise
# of that rounding: an fp64 simulation of the method gives 1.1 - 1.8 % RMS
# relative to the output on the tiny, edge and full-size FP8 shapes with
# outliers, and 2.5 - 3.5 % with P rounded to two mantissa bits instead of
# three (tests/test_fp8_bound.py), so 2.5 %.
BF16_MAX_ABS = 1e-2
BF16_MEAN_ABS = 1e-3
BF16_REL_RMS = 1e-2
FP8_MAX_ABS = 6e-2
FP8_REL_RMS = 2.5e-2


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def device_inputs(inp):
    return dict(q=dev_bf16(inp.q), k=dev_bf16(inp.k), v=dev_bf16(inp.v),
                q_norm_w=torch.from_numpy(inp.w_q).cuda(), k_norm_w=torch.from_numpy(inp.w_k).cuda(),
                pos_ids=torch.from_numpy(inp.pos).cuda())


def gather_rows(out_bnhd: np.ndarray, rows: np.ndarray) -> np.ndarray:
    return out_bnhd[rows[:, 0], rows[:, 2], rows[:, 1], :]


def compare(got: np.ndarray, want: np.ndarray, max_abs: float, mean_abs: float = None,
            rel_rms: float = None, what: str = ""):
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite output" % what
    err = np.abs(got - want)
    stats = dict(max_abs=float(err.max()), mean_abs=float(err.mean()),
                 rel_rms=float(np.sqrt((err ** 2).mean() / max((want ** 2).mean(), 1e-300))))
    msg = "%s: %s" % (what, stats)
    assert stats["max_abs"] <= max_abs, msg
    if mean_abs is not None:
        assert stats["mean_abs"] <= mean_abs, msg
    if rel_rms is not None:
        assert stats["rel_rms"] <= rel_rms, msg
    return stats


def v8t_token_order(v8t: np.ndarray) -> np.ndarray:
    """V^T codes of the plain FP8 prologue with the columns back in token order.
    Within every 8 columns the prologue stores tokens 0, 2, 4, 6, 1, 3, 5, 7: the
    key order of the FP8 attention's P.V MMA, whose softmax threads each hold the
    even or the odd keys of a row.  Column 8g + 4p + b holds token 8g + 2b + p."""
    col = np.arange(v8t.shape[-1])
    token = 8 * (col // 8) + 2 * (col % 4) + (col % 8) // 4
    out = np.empty_like(v8t)
    out[..., token] = v8t
    return out
