"""QKV projection with the fused QK-norm + RoPE epilogue against the fp64
oracle (GPU).

The GPU accumulates x W^T in fp32 over d_model products, applies bias, the
RMSNorm and the rotation in fp32 and rounds once to bf16; the oracle does the
same arithmetic in fp64.  So every output element must be within half a bf16
ulp (2^-9 relative) plus the fp32 error, bounded here by 2^-8 |ref| + 1e-5.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import dev_bf16, host_f64, v8t_token_order

pytestmark = pytest.mark.gpu

import diffusion_transformer_joint_txt_b300 as fa  # noqa: E402


def _run(w, inp, bias=True, handle=None):
    attn = handle or fa.FluxAttention(w.batch, w.heads, w.tokens)
    x = dev_bf16(inp.x)
    wt = dev_bf16(inp.w)
    b = torch.from_numpy(inp.bias).cuda() if bias else None
    qn, kn, v = attn.qkv(x, wt, b, w.txt_len, w.img_h, w.img_w, w.ref_h, w.ref_w,
                         torch.from_numpy(inp.w_q).cuda(), torch.from_numpy(inp.w_k).cuda())
    assert attn.sync_status() == 0
    return attn, qn, kn, v


def _check(got, want, what):
    err = np.abs(got - want)
    bound = 2.0 ** -8 * np.abs(want) + 1e-5
    bad = err > bound
    assert not bad.any(), "%s: %d of %d outside 2^-8 |ref| + 1e-5 (worst excess %.3e)" % (
        what, int(bad.sum()), bad.size, float((err - bound).max()))


def _compare(w, inp, qn, kn, v, rows=None, bias=True):
    B, N, H = w.batch, w.tokens, w.heads
    oq, ok, ov = oracle.qkv_rows(inp.x, inp.w, inp.bias if bias else None, N, inp.pos, inp.w_q, inp.w_k, H,
                                 rows=rows)
    m = np.arange(B * N) if rows is None else rows
    b, n = m // N, m % N
    gq = host_f64(qn)[b, :, n, :]          # [R, H, 128]
    gk = host_f64(kn)[b, :, n, :]
    gv = host_f64(v)[b, n, :, :]
    _check(gq, oq, "Q'")
    _check(gk, ok, "K'")
    _check(gv, ov, "V")


@pytest.mark.parametrize("B,H,txt,ih,iw,rh,rw,D,bias", [
    (2, 2, 7, 5, 9, 0, 0, 256, True),       # N = 52: one partial token tile
    (1, 3, 64, 16, 16, 2, 3, 192, False),   # odd H: a 256-wide tile straddles the Q/K and K/V boundaries
    (2, 4, 100, 10, 12, 0, 0, 512, True),   # 440 tokens: several token tiles per weight tile
])
def test_qkv_every_element(B, H, txt, ih, iw, rh, rw, D, bias):
    w = synthetic.Workload("qkv", B, H, txt, ih, iw, rh, rw)
    inp = synthetic.make_qkv_inputs(w, D, seed=B * 10 + H)
    _, qn, kn, v = _run(w, inp, bias)
    _compare(w, inp, qn, kn, v, bias=bias)


def test_qkv_flux_1024_sampled_rows():
    w = synthetic.WORKLOADS["flux_1024_4608"]
    inp = synthetic.make_qkv_inputs(w)
    _, qn, kn, v = _run(w, inp)
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, 127, 128, 511, 512, 4607], rng.integers(0, w.tokens, 40)]))
    _compare(w, inp, qn, kn, v, rows=rows)


def test_qkv_then_attend_matches_forward_on_the_projection():
    """flux_attn_qkv + flux_attn_attend equals flux_attn_forward applied to the
    (unnormalised) projection computed by torch on the GPU: the fused epilogue
    and the prologue kernel agree."""
    w = synthetic.Workload("qkv_chain", 1, 2, 30, 8, 8)
    inp = synthetic.make_qkv_inputs(w, 256, seed=7)
    attn, qn, kn, v = _run(w, inp)
    out = attn.attend(qn, kn, v)
    x = dev_bf16(inp.x).float()
    y = x @ dev_bf16(inp.w).float().T + torch.from_numpy(inp.bias).cuda()
    H, N = w.heads, w.tokens
    q, k, vv = (y[:, i * H * 128:(i + 1) * H * 128].reshape(1, N, H, 128).to(torch.bfloat16) for i in range(3))
    ref = attn.forward(q.contiguous(), k.contiguous(), vv.contiguous(), w.txt_len, w.img_h, w.img_w, 0, 0,
                       torch.from_numpy(inp.w_q).cuda(), torch.from_numpy(inp.w_k).cuda())
    assert attn.sync_status() == 0
    diff = (out.float() - ref.float()).abs().max().item()
    assert diff <= 2e-2, diff       # only the bf16 rounding of the projection before the prologue differs


def test_qkv_rejects_bad_arguments():
    w = synthetic.Workload("qkv_bad", 1, 2, 8, 2, 4)
    inp = synthetic.make_qkv_inputs(w, 128)
    attn = fa.FluxAttention(1, 2, w.tokens)
    x, wt = dev_bf16(inp.x), dev_bf16(inp.w)
    ones = torch.ones(128, device="cuda")
    hm = torch.empty((1, 2, w.tokens, 128), dtype=torch.bfloat16, device="cuda")
    vv = torch.empty((1, w.tokens, 2, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FluxAttnError) as e:      # d_model not a multiple of 64
        fa.flux_attn_qkv(attn.handle, x, wt, None, 96, 8, 2, 4, 0, 0, None, ones, ones, hm, hm.clone(), vv)
    assert e.value.status == fa.FLUX_ATTN_ERR_UNSUPPORTED
    with pytest.raises(fa.FluxAttnError) as e:      # outputs alias
        fa.flux_attn_qkv(attn.handle, x, wt, None, 128, 8, 2, 4, 0, 0, None, ones, ones, hm, hm, vv)
    assert e.value.status == fa.FLUX_ATTN_ERR_INVALID_ARG
    f8 = fa.FluxAttention(1, 2, w.tokens, precision="fp8")
    with pytest.raises(fa.FluxAttnError) as e:
        fa.flux_attn_qkv(f8.handle, x, wt, None, 128, 8, 2, 4, 0, 0, None, ones, ones, hm, hm.clone(), vv)
    assert e.value.status == fa.FLUX_ATTN_ERR_UNSUPPORTED


def test_forward_hidden_equals_qkv_then_attend():
    w = synthetic.Workload("hidden", 2, 3, 20, 9, 13, 2, 2)
    inp = synthetic.make_qkv_inputs(w, 384, seed=9)
    attn, qn, kn, v = _run(w, inp)
    want = attn.attend(qn, kn, v)
    got = attn.forward_hidden(dev_bf16(inp.x), dev_bf16(inp.w), torch.from_numpy(inp.bias).cuda(), w.txt_len,
                              w.img_h, w.img_w, w.ref_h, w.ref_w, torch.from_numpy(inp.w_q).cuda(),
                              torch.from_numpy(inp.w_k).cuda())
    assert attn.sync_status() == 0
    assert torch.equal(got, want)


def test_qkv_alternating_geometry_no_sync():
    """The GEMM starts before its (cos, sin) table kernel has finished and
    only its epilogue waits for it: two geometries with the same token count
    alternate step after step without host synchronisation, and each step's
    Q', K' must equal those computed with a sync after the table kernel, bit
    for bit (a stale table would rotate by the other geometry's angles)."""
    w = synthetic.Workload("qkv_geo", 1, 4, 512, 32, 32, 0, 0)          # N = 1536
    inp = synthetic.make_qkv_inputs(w, d_model=256, seed=31)
    geos = [(512, 32, 32, 0, 0), (256, 16, 64, 8, 32)]                  # 512 + 1024 = 256 + 1024 + 256
    assert len({g[0] + g[1] * g[2] + g[3] * g[4] for g in geos}) == 1
    attn = fa.FluxAttention(w.batch, w.heads, w.tokens)
    x, wt = dev_bf16(inp.x), dev_bf16(inp.w)
    b = torch.from_numpy(inp.bias).cuda()
    wq, wk = torch.from_numpy(inp.w_q).cuda(), torch.from_numpy(inp.w_k).cuda()
    qn, kn, v = attn.qkv(x, wt, b, *geos[0], wq, wk)
    refs = []
    for g in geos:
        attn.qkv(x, wt, b, *g, wq, wk, qn=qn, kn=kn, v=v)
        torch.cuda.synchronize()
        refs.append((qn.clone(), kn.clone()))
    assert not torch.equal(refs[0][0], refs[1][0])
    steps = 10
    snaps = []
    for i in range(steps):
        attn.qkv(x, wt, b, *geos[i % 2], wq, wk, qn=qn, kn=kn, v=v)
        snaps.append((qn.clone(), kn.clone()))
    torch.cuda.synchronize()
    assert attn.sync_status() == 0
    bad = [i for i in range(steps) if not (torch.equal(snaps[i][0], refs[i % 2][0]) and
                                           torch.equal(snaps[i][1], refs[i % 2][1]))]
    assert not bad, "steps with another geometry's rotation: %s" % bad


# ------------------------------------------------------------------ FP8 codes

_DECODE = None


def _decode():
    global _DECODE
    if _DECODE is None:
        _DECODE = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    return _DECODE


def _codes_close(got, want, x, scale, what):
    """E4M3 codes of the GPU (from its bf16 Q', K', V and a scale from their bf16
    amax) against the oracle's (fp64 values x, fp64 amax).  A code may differ
    only by one step, only where x / scale lies within 2^-7 (relative) of the
    midpoint between the two codes -- the bf16 rounding before the codes can
    move a value across it -- and for at most 5 % of the codes."""
    diff = got != want
    assert diff.mean() <= 0.05, "%s: %.3f of the codes differ" % (what, diff.mean())
    if not diff.any():
        return
    t = _decode()
    a, b = t[got[diff]], t[want[diff]]
    assert np.all(np.sign(a) * np.sign(b) >= 0), what
    mid = 0.5 * (a + b)
    q = x[diff] / scale
    step = np.abs(a - b)
    assert np.all(step <= np.maximum(np.abs(b), 2.0 ** -6) * 2.0 ** -2), what   # neighbours (or the two next to 0)
    assert np.all(np.abs(q - mid) <= 2.0 ** -7 * np.maximum(np.abs(mid), 2.0 ** -9) + 2.0 ** -10), what


@pytest.mark.parametrize("B,H,txt,ih,iw,rh,rw,D", [
    (2, 3, 7, 5, 9, 0, 0, 256),      # N = 52, B = 2: a token tile spans both batch rows
    (1, 2, 100, 10, 12, 2, 3, 192),  # N = 226 with a reference stream
])
def test_qkv_fp8_codes_and_scales(B, H, txt, ih, iw, rh, rw, D):
    """The FP8 QKV projection's codes and scales against the oracle's
    projection quantised per (b, h) by the oracle (reading R5)."""
    w = synthetic.Workload("qkv8", B, H, txt, ih, iw, rh, rw)
    inp = synthetic.make_qkv_inputs(w, D, seed=B * 13 + H)
    attn = fa.FluxAttention(B, H, w.tokens, precision="fp8")
    x, wt = dev_bf16(inp.x), dev_bf16(inp.w)
    b = torch.from_numpy(inp.bias).cuda()
    wq, wk = torch.from_numpy(inp.w_q).cuda(), torch.from_numpy(inp.w_k).cuda()
    q8, k8, v8t, scales = attn.qkv_fp8(x, wt, b, w.txt_len, w.img_h, w.img_w, w.ref_h, w.ref_w, wq, wk)
    out = attn.attend_fp8(q8, k8, v8t, scales)
    full = attn.forward_hidden(x, wt, b, w.txt_len, w.img_h, w.img_w, w.ref_h, w.ref_w, wq, wk)
    assert attn.sync_status() == 0
    assert torch.equal(out, full)
    N = w.tokens
    oq, ok, ov = oracle.qkv_rows(inp.x, inp.w, inp.bias, N, inp.pos, inp.w_q, inp.w_k, H)   # [B N, H, 128]
    q8h, k8h, v8h, sch = (t.cpu().numpy() for t in (q8, k8, v8t, scales))
    v8h = v8t_token_order(v8h)
    for bb in range(B):
        for hh in range(H):
            for t, (vals, codes) in enumerate(((oq, q8h[bb, hh]), (ok, k8h[bb, hh]), (ov, v8h[bb, hh, :, :N].T))):
                xv = vals[bb * N:(bb + 1) * N, hh, :]
                want, scale = oracle.fp8_quantize(xv)
                np.testing.assert_allclose(sch[bb, hh, t], scale, rtol=2.0 ** -8)
                _codes_close(codes, want, xv, scale, "(%d, %d) tensor %d" % (bb, hh, t))
