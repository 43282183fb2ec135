"""Seeded synthetic workloads for the joint text/image attention path.

This module is shared by the oracle-side tests and the CUDA-side tests and
bench.  It holds only random draws, the bf16 rounding of those draws and the
token-geometry bookkeeping (how many text / image / reference tokens, and the
3-axis integer position ids each token carries).  None of the attention
arithmetic (normalisation, rotation, softmax) lives here.

Workload shapes follow the FLUX-style denoising steps described in
"Speed up image generation with FLUX 3 Image Klein on NVIDIA Blackwell GPUs"
(NVIDIA developer blog, section "FLUX 3 inference with TensorRT LLM
VisualGen": text, noisy target image and optional reference image streams are
concatenated and attend jointly) and the 1024x1024 -> 64x64 packed latent of
"FLUX.1-dev latency optimisation roundup" (parameter table).

Recipe (the same for every workload):
  * numpy.random.default_rng(seed), seed 0 by default;
  * draw order q, k, v (each [B, N, H, D] standard normal, float32), then
    w_q, w_k (each [D], 1 + 0.1 * N(0, 1), kept as float32);
  * workloads with outliers draw, right after each of q, k, v, a uniform
    mask with p = 0.01 and multiply the masked entries by 8;
  * q, k, v are rounded to bf16 with round-to-nearest-even (stored as the
    uint16 bit pattern); the weights stay float32;
  * position ids per token: text (0, 0, 0), target image (0, row, col),
    reference image (1, row, col), row-major over each grid.

QKV-projection inputs (make_qkv_inputs): hidden states x [B, N, D] standard
normal, then the stacked weight W [3 H d, D] and bias [3 H d] drawn like a
freshly initialised linear layer (uniform on +-1/sqrt(D)), then w_q, w_k as
above; x and W are rounded to bf16, the bias stays float32.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np

HEAD_DIM = 128
AXES_DIM = (16, 56, 56)
ROPE_THETA = 10000.0
RMS_EPS = 1e-6


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    txt_len: int
    img_h: int
    img_w: int
    ref_h: int = 0
    ref_w: int = 0
    precision: str = "bf16"        # "bf16" or "fp8"
    outliers: bool = False
    head_dim: int = HEAD_DIM
    vc_repair_budget: float = 0.0  # FP8 with VC-Attention repair when > 0
    sol_tau: float = 0.0           # block-sparse Sol-Attention threshold when > 0

    @property
    def tokens(self) -> int:
        return self.txt_len + self.img_h * self.img_w + self.ref_h * self.ref_w

    @property
    def flops(self) -> int:
        """4 * B * H * N^2 * d: two N x N x d contractions of 2 flops per MAC."""
        return 4 * self.batch * self.heads * self.tokens ** 2 * self.head_dim

    def describe(self) -> Dict[str, object]:
        return {"workload": self.name, "batch": self.batch, "heads": self.heads,
                "head_dim": self.head_dim, "txt_len": self.txt_len,
                "img": [self.img_h, self.img_w], "ref": [self.ref_h, self.ref_w],
                "tokens": self.tokens, "precision": self.precision}


# The five workloads: a tiny case, FLUX-dev 1024^2, FLUX 2048^2, image-to-image
# with a 2048^2 reference, and the FP8 classifier-free-guidance pair at 2048^2.
WORKLOADS: Dict[str, Workload] = {
    "tiny_320": Workload("tiny_320", 1, 2, 64, 16, 16),
    "flux_1024_4608": Workload("flux_1024_4608", 1, 24, 512, 64, 64),
    "flux_2048_16896": Workload("flux_2048_16896", 1, 24, 512, 128, 128),
    "i2i_2048_33280": Workload("i2i_2048_33280", 1, 24, 512, 128, 128, 128, 128),
    "fp8_cfg_2048_16896": Workload("fp8_cfg_2048_16896", 2, 24, 512, 128, 128,
                                   precision="fp8", outliers=True),
    # the same pair with the VC-Attention repair budget of the page's configuration
    "vc_fp8_cfg_2048_16896": Workload("vc_fp8_cfg_2048_16896", 2, 24, 512, 128, 128,
                                      precision="fp8", outliers=True, vc_repair_budget=0.005),
    # FLUX 2048^2 with the block-sparse attention at the page's tau
    "sol_flux_2048_16896": Workload("sol_flux_2048_16896", 1, 24, 512, 128, 128, sol_tau=1.0),
}
WORKLOAD_ORDER = ["tiny_320", "flux_1024_4608", "flux_2048_16896",
                  "i2i_2048_33280", "fp8_cfg_2048_16896"]


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits.

    Inputs are finite draws, so no NaN handling is needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def position_ids(txt_len: int, img_h: int, img_w: int, ref_h: int = 0, ref_w: int = 0) -> np.ndarray:
    """[N, 3] int32 ids: text (0,0,0), image (0,r,c), reference (1,r,c)."""
    parts = [np.zeros((txt_len, 3), np.int32)]
    if img_h * img_w:
        r, c = np.meshgrid(np.arange(img_h), np.arange(img_w), indexing="ij")
        parts.append(np.stack([np.zeros(img_h * img_w, np.int64), r.ravel(), c.ravel()], 1).astype(np.int32))
    if ref_h * ref_w:
        r, c = np.meshgrid(np.arange(ref_h), np.arange(ref_w), indexing="ij")
        parts.append(np.stack([np.ones(ref_h * ref_w, np.int64), r.ravel(), c.ravel()], 1).astype(np.int32))
    return np.ascontiguousarray(np.concatenate(parts, 0), dtype=np.int32)


@dataclasses.dataclass
class Inputs:
    workload: Workload
    q: np.ndarray      # uint16 bf16 bits [B, N, H, D]
    k: np.ndarray
    v: np.ndarray
    w_q: np.ndarray    # float32 [D]
    w_k: np.ndarray
    pos: np.ndarray    # int32 [N, 3]


def _draw(rng: np.random.Generator, shape, outliers: bool) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if outliers:
        mask = rng.random(shape, dtype=np.float32) < np.float32(0.01)
        x[mask] *= np.float32(8.0)
    return bf16_bits_from_f32(x)


def make_inputs(w: Workload, seed: int = 0, tokens_override: Optional[tuple] = None) -> Inputs:
    """Draw the seeded inputs of workload ``w`` (see the module docstring)."""
    txt, ih, iw, rh, rw = tokens_override or (w.txt_len, w.img_h, w.img_w, w.ref_h, w.ref_w)
    n = txt + ih * iw + rh * rw
    shape = (w.batch, n, w.heads, w.head_dim)
    rng = np.random.default_rng(seed)
    q = _draw(rng, shape, w.outliers)
    k = _draw(rng, shape, w.outliers)
    v = _draw(rng, shape, w.outliers)
    w_q = (1.0 + 0.1 * rng.standard_normal(w.head_dim)).astype(np.float32)
    w_k = (1.0 + 0.1 * rng.standard_normal(w.head_dim)).astype(np.float32)
    return Inputs(w, q, k, v, w_q, w_k, position_ids(txt, ih, iw, rh, rw))


def sample_rows(w: Workload, n_tokens: int, per_head: int, seed: int = 1) -> np.ndarray:
    """Seeded (b, h, n) query rows for sampled parity at full size.

    Every (b, h) gets ``per_head`` random rows plus the boundary rows: first
    and last text, image and reference tokens, both sides of every 128-row
    tile edge that falls inside a stream boundary, and row N-1.
    """
    rng = np.random.default_rng(seed)
    txt = w.txt_len
    img = w.img_h * w.img_w
    edges = {0, n_tokens - 1}
    if txt:
        edges |= {txt - 1, min(txt, n_tokens - 1)}
    if img:
        edges |= {txt, txt + img - 1}
    if w.ref_h * w.ref_w:
        edges |= {txt + img, n_tokens - 1}
    for t in (127, 128, 255, 256):
        if t < n_tokens:
            edges.add(t)
    edges = sorted(e for e in edges if 0 <= e < n_tokens)
    rows = []
    for b in range(w.batch):
        for h in range(w.heads):
            picks = set(edges) | set(rng.integers(0, n_tokens, per_head).tolist())
            rows.extend((b, h, n) for n in sorted(picks))
    return np.asarray(rows, dtype=np.int64)


@dataclasses.dataclass
class QKVInputs:
    workload: Workload
    d_model: int
    x: np.ndarray      # uint16 bf16 bits [B * N, D]
    w: np.ndarray      # uint16 bf16 bits [3 H d, D]
    bias: np.ndarray   # float32 [3 H d]
    w_q: np.ndarray    # float32 [d]
    w_k: np.ndarray
    pos: np.ndarray    # int32 [N, 3]


def make_qkv_inputs(w: Workload, d_model: Optional[int] = None, seed: int = 0) -> QKVInputs:
    """Seeded inputs of the QKV projection for workload ``w``; the hidden size
    defaults to H * d (3072 for the FLUX workloads)."""
    D = d_model or w.heads * w.head_dim
    n = w.tokens
    F = 3 * w.heads * w.head_dim
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((w.batch * n, D), dtype=np.float32)
    lim = np.float32(1.0 / np.sqrt(D))
    wt = rng.uniform(-lim, lim, (F, D)).astype(np.float32)
    bias = rng.uniform(-lim, lim, F).astype(np.float32)
    w_q = (1.0 + 0.1 * rng.standard_normal(w.head_dim)).astype(np.float32)
    w_k = (1.0 + 0.1 * rng.standard_normal(w.head_dim)).astype(np.float32)
    return QKVInputs(w, D, bf16_bits_from_f32(x), bf16_bits_from_f32(wt), bias, w_q, w_k,
                     position_ids(w.txt_len, w.img_h, w.img_w, w.ref_h, w.ref_w))
