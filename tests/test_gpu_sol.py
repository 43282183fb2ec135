"""Sol-Attention (block-sparse joint attention) through the C ABI against the
fp64 oracle (GPU).

"Speed up image generation with FLUX 3 Image Klein on NVIDIA Blackwell GPUs",
section "Quantized and sparse attention": Sol-Attention with tau 1.0, dense
until the timestep falls to 0.96 (reading R8 of the oracle: 128-token
blocks, pooled-mean block masses weighted by block size, keep mu >= tau / nb
plus the block of largest mass).

What is compared:
  * the block mask (index work): equal to the oracle's, except for blocks
    whose oracle mass lies within 1e-4 (relative) of the threshold -- the GPU
    decides on its bf16 Q', K' in fp32, the oracle on fp64;
  * the output of every query block whose mask row agrees: BF16 tolerances
    (max-abs 1e-2, mean-abs 1e-3, relative RMS 1 %) against the oracle's
    sparse attention;
  * a tau small enough to keep every block gives the dense kernel's output bit
    for bit (the same blocks in the same order), and the timestep gate runs
    the dense kernel above the cutoff.
Inputs: seeded N(0, 1) bf16, plus a planted direction shared by some query and
key blocks so that the masks hold structure besides noise.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import BF16_MAX_ABS, BF16_MEAN_ABS, BF16_REL_RMS, compare, device_inputs, gather_rows

pytestmark = pytest.mark.gpu

import diffusion_transformer_joint_txt_b300 as fa  # noqa: E402


def _f32(x):
    return float(np.float32(x))


def _geom(w):
    return w.txt_len, w.img_h, w.img_w, w.ref_h, w.ref_w


def _inputs(w, seed, plant=True):
    inp = synthetic.make_inputs(w, seed=seed)
    if plant:   # query blocks 1, 3 and key blocks 2, 5 (where present) share a direction
        rng = np.random.default_rng(seed + 100)
        n = w.tokens
        q = synthetic.bf16_bits_to_f32(inp.q).copy()
        k = synthetic.bf16_bits_to_f32(inp.k).copy()
        for hh in range(w.heads):
            dirn = rng.standard_normal(128).astype(np.float32) * 2.0
            for qb in (1, 3):
                q[:, qb * 128:min(n, qb * 128 + 128), hh] += dirn
            for kb in (2, 5):
                k[:, kb * 128:min(n, kb * 128 + 128), hh] += dirn
        inp.q[...] = synthetic.bf16_bits_from_f32(q)
        inp.k[...] = synthetic.bf16_bits_from_f32(k)
    return inp


def _check_mask(keep, inp, w, tau):
    """GPU masks [B, H, nb, nb] against the oracle's; returns the mask rows
    (b, h, query block) that agree."""
    agree = np.zeros(keep.shape[:3], bool)
    nb = keep.shape[-1]
    for b in range(w.batch):
        for h in range(w.heads):
            want, mass = oracle.sol_mask(inp.q, inp.k, inp.pos, inp.w_q, inp.w_k, tau, b, h)
            got = keep[b, h].astype(bool)
            diff = got != want
            thr = tau / nb
            near = np.abs(mass - thr) <= 1e-4 * thr
            assert np.all(near[diff]), ("head", b, h, np.argwhere(diff & ~near)[:5])
            agree[b, h] = ~diff.any(axis=1)
    return agree


CASES = [
    # B, H, txt, img_h, img_w, ref_h, ref_w, tau
    (1, 2, 64, 16, 16, 0, 0, 1.0),      # N = 320: three blocks, the last ragged
    (2, 3, 40, 20, 30, 4, 9, 1.0),      # N = 676 with a reference stream, six blocks
    (1, 2, 100, 24, 40, 0, 0, 1.5),     # N = 1060, nine blocks, a sparser tau
    (1, 4, 7, 5, 9, 0, 0, 1.0),         # N = 52: one block (kept: the block of largest mass)
]


@pytest.mark.parametrize("B,H,txt,ih,iw,rh,rw,tau", CASES)
def test_sol_mask_and_rows(B, H, txt, ih, iw, rh, rw, tau):
    tau = _f32(tau)
    w = synthetic.Workload("sol", B, H, txt, ih, iw, rh, rw)
    inp = _inputs(w, seed=B * 17 + txt)
    d = device_inputs(inp)
    attn = fa.FluxAttention(B, H, w.tokens, sol_tau=tau, sol_disabled_until_timestep=0.96)
    qn, kn = attn.prologue(d["q"], d["k"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    keep = attn.sol_mask(qn, kn)
    out = attn.attend_sol(qn, kn, d["v"], keep)
    full = attn.forward_sol(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"], timestep=0.5)
    assert attn.sync_status() == 0
    assert torch.equal(out, full)
    keep_h = keep.cpu().numpy()
    assert np.all(keep_h.sum(-1) >= 1)
    agree = _check_mask(keep_h, inp, w, tau)
    rows = np.array([(b, h, n) for b in range(B) for h in range(H) for n in range(w.tokens)
                     if agree[b, h, n // 128]], np.int64)
    assert len(rows) >= 0.9 * B * H * w.tokens
    want = oracle.sol_attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k, tau, rows=rows)
    got = gather_rows(out.float().cpu().numpy().astype(np.float64), rows)
    compare(got, want, BF16_MAX_ABS, BF16_MEAN_ABS, BF16_REL_RMS, what="sol N=%d tau=%g" % (w.tokens, tau))
    # and it is not the dense result where blocks were dropped
    if (keep_h == 0).any():
        dense = oracle.attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k, rows=rows)
        assert np.abs(dense - want).max() > 1e-2


def test_sol_keeping_every_block_is_the_dense_kernel():
    w = synthetic.Workload("sol_all", 1, 3, 64, 16, 20)            # N = 384
    inp = _inputs(w, seed=5)
    d = device_inputs(inp)
    attn = fa.FluxAttention(1, 3, w.tokens, sol_tau=1e-20)
    qn, kn = attn.prologue(d["q"], d["k"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    keep = attn.sol_mask(qn, kn)
    sparse = attn.attend_sol(qn, kn, d["v"], keep)
    dense = attn.attend(qn, kn, d["v"])
    assert attn.sync_status() == 0
    assert bool((keep == 1).all())
    assert torch.equal(sparse, dense)


def test_sol_one_block_per_query_block():
    """A tau above nb keeps only each query block's block of largest mass."""
    tau = _f32(50.0)
    w = synthetic.Workload("sol_one", 1, 2, 40, 20, 30)              # N = 640, five blocks
    inp = _inputs(w, seed=8)
    d = device_inputs(inp)
    attn = fa.FluxAttention(1, 2, w.tokens, sol_tau=tau)
    qn, kn = attn.prologue(d["q"], d["k"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    keep = attn.sol_mask(qn, kn)
    out = attn.attend_sol(qn, kn, d["v"], keep)
    assert attn.sync_status() == 0
    keep_h = keep.cpu().numpy()
    assert np.all(keep_h.sum(-1) == 1)
    agree = _check_mask(keep_h, inp, w, tau)
    assert agree.all()
    want = oracle.sol_attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k, tau)
    compare(out.float().cpu().numpy().astype(np.float64), want, BF16_MAX_ABS, BF16_MEAN_ABS, BF16_REL_RMS,
            what="sol one block")


def test_sol_timestep_gate_runs_dense_above_the_cutoff():
    w = synthetic.Workload("sol_gate", 1, 2, 64, 16, 16)
    inp = _inputs(w, seed=9)
    d = device_inputs(inp)
    attn = fa.FluxAttention(1, 2, w.tokens, sol_tau=1.0, sol_disabled_until_timestep=0.96)
    early = attn.forward_sol(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"], timestep=0.98)
    dense = attn.forward(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    late = attn.forward_sol(d["q"], d["k"], d["v"], *_geom(w), d["q_norm_w"], d["k_norm_w"], timestep=0.96)
    assert attn.sync_status() == 0
    assert torch.equal(early, dense)
    assert not torch.equal(late, dense)


def test_sol_full_size_sampled_rows():
    """FLUX 2048^2 (N = 16896, 132 blocks) at the page's tau 1.0: mask of every
    head, then 16 random rows per head plus the boundary rows."""
    tau = _f32(1.0)
    w = synthetic.WORKLOADS["flux_2048_16896"]
    inp = synthetic.make_inputs(w)
    d = device_inputs(inp)
    attn = fa.FluxAttention(w.batch, w.heads, w.tokens, sol_tau=tau)
    qn, kn = attn.prologue(d["q"], d["k"], *_geom(w), d["q_norm_w"], d["k_norm_w"])
    keep = attn.sol_mask(qn, kn)
    out = attn.attend_sol(qn, kn, d["v"], keep)
    assert attn.sync_status() == 0
    keep_h = keep.cpu().numpy()
    agree = _check_mask(keep_h, inp, w, tau)
    rows = synthetic.sample_rows(w, w.tokens, 16)
    rows = rows[agree[rows[:, 0], rows[:, 1], rows[:, 2] // 128]]
    want = oracle.sol_attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k, tau, rows=rows)
    got = gather_rows(out.float().cpu().numpy().astype(np.float64), rows)
    compare(got, want, BF16_MAX_ABS, BF16_MEAN_ABS, BF16_REL_RMS, what="sol " + w.name)


def test_sol_handle_rules():
    with pytest.raises(fa.FluxAttnError) as e:
        fa.FluxAttention(1, 2, 256, precision="fp8", sol_tau=1.0)
    assert e.value.status == fa.FLUX_ATTN_ERR_INVALID_ARG
    plain = fa.FluxAttention(1, 2, 256)
    x = torch.zeros((1, 2, 256, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FluxAttnError) as e:
        plain.sol_mask(x, x)
    assert e.value.status == fa.FLUX_ATTN_ERR_INVALID_ARG
