"""The allocation-free forward against the ordinary forward (GPU).

Some callers of this library must not allocate device memory while they run:
engines that reserve and plan all device memory once at start-up and forbid
later allocations, plugin hosts that give a plugin only the buffers it
declared, and latency-critical callers that cannot take the device-wide
synchronisation an allocation may cause.  flux_attn_forward_noalloc serves
them: no handle, no allocation, its scratch in a fixed device array shared by
every call.  These checks call it through the C ABI and compare it with
flux_attn_forward on the same inputs, on two calls in a row (the second one
finds the first one's data still in the scratch).

This file is collected last so that a run that stops at its first failure has
already run every other test; it passes alone in a fresh process as well.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import BF16_MAX_ABS, BF16_MEAN_ABS, BF16_REL_RMS, compare, device_inputs, host_f64

pytestmark = pytest.mark.gpu

import diffusion_transformer_joint_txt_b300 as fa  # noqa: E402

# two different problems, one right after the other
CALLS = [
    (synthetic.Workload("noalloc_a", 1, 4, 77, 20, 24), 11),         # N = 557
    (synthetic.Workload("noalloc_b", 2, 3, 13, 11, 17, 3, 4), 12),   # N = 212, with a reference stream
]


def _geom(w):
    return (w.txt_len, w.img_h, w.img_w, w.ref_h, w.ref_w)


def _prepare(w, seed):
    inp = synthetic.make_inputs(w, seed=seed)
    d = device_inputs(inp)
    cfg = fa.make_config(w.batch, w.heads, w.tokens)
    ref = torch.empty_like(d["q"])
    h = fa.flux_attn_create(w.batch, w.heads, w.tokens)
    fa.flux_attn_forward(h, d["q"], d["k"], d["v"], *_geom(w), None, d["q_norm_w"], d["k_norm_w"], ref)
    assert fa.flux_attn_sync_status(h) == 0
    fa.flux_attn_destroy(h)
    return d, cfg, ref


def test_noalloc_matches_forward_on_two_calls_in_a_row():
    prepared = [(w, *_prepare(w, seed)) for w, seed in CALLS]
    err_word = torch.full((4,), 7, dtype=torch.int32, device="cuda")
    outs = [torch.full_like(ref, float("nan")) for _, _, _, ref in prepared]
    for (w, d, cfg, ref), out in zip(prepared, outs):
        fa.flux_attn_forward_noalloc(cfg, d["q"], d["k"], d["v"], *_geom(w), None, d["q_norm_w"], d["k_norm_w"],
                                     out, device_error=err_word)
    torch.cuda.synchronize()
    assert int(err_word[0].item()) == 0
    for (w, d, cfg, ref), out in zip(prepared, outs):
        assert torch.equal(out, ref)   # the same kernels on the same inputs


def test_noalloc_matches_the_oracle():
    """The second problem (B = 2, a reference stream) against the fp64 oracle,
    every row, with the tolerances of the other BF16 tests."""
    w, seed = CALLS[1]
    inp = synthetic.make_inputs(w, seed=seed)
    d = device_inputs(inp)
    cfg = fa.make_config(w.batch, w.heads, w.tokens)
    out = torch.empty_like(d["q"])
    fa.flux_attn_forward_noalloc(cfg, d["q"], d["k"], d["v"], *_geom(w), None, d["q_norm_w"], d["k_norm_w"], out)
    torch.cuda.synchronize()
    want = oracle.attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k)
    compare(host_f64(out), want, BF16_MAX_ABS, BF16_MEAN_ABS, BF16_REL_RMS, what="noalloc vs oracle " + w.name)


def test_noalloc_reports_a_device_timeout_and_clears_it():
    """A call whose bounded wait runs out (the forced-timeout debug flag: the
    attention kernel waits on a barrier nothing signals, for about a second)
    reports a nonzero device error word; the next clean call clears the word
    in the shared scratch and gives the ordinary forward's result again."""
    w, seed = CALLS[0]
    d, cfg, ref = _prepare(w, seed)
    bad = fa.make_config(w.batch, w.heads, w.tokens, debug_flags=fa.FLUX_ATTN_DEBUG_FORCE_TIMEOUT)
    err_word = torch.zeros((4,), dtype=torch.int32, device="cuda")
    out = torch.empty_like(ref)
    fa.flux_attn_forward_noalloc(bad, d["q"], d["k"], d["v"], *_geom(w), None, d["q_norm_w"], d["k_norm_w"],
                                 out, device_error=err_word)
    torch.cuda.synchronize()
    assert int(err_word[0].item()) != 0
    err_word.fill_(7)
    fa.flux_attn_forward_noalloc(cfg, d["q"], d["k"], d["v"], *_geom(w), None, d["q_norm_w"], d["k_norm_w"],
                                 out, device_error=err_word)
    torch.cuda.synchronize()
    assert int(err_word[0].item()) == 0
    assert torch.equal(out, ref)


def test_noalloc_allocates_nothing():
    """Neither the device's free memory nor torch's allocator statistics move
    across three calls.  Free memory catches fresh device allocations (a
    cudaMalloc of the library's own); it cannot see an allocation served from
    memory a stream-ordered pool had already reserved, so the docstring of the
    entry point (no cudaMalloc, cudaFree or allocating library call) is the
    contract and this is its check on the device."""
    w, seed = CALLS[0]
    d, cfg, ref = _prepare(w, seed)
    out = torch.empty_like(ref)
    args = (cfg, d["q"], d["k"], d["v"], *_geom(w), None, d["q_norm_w"], d["k_norm_w"], out)
    fa.flux_attn_forward_noalloc(*args)            # the first call on this device may do its set-up
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    stats_before = torch.cuda.memory_stats()
    for _ in range(3):
        fa.flux_attn_forward_noalloc(*args)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    stats_after = torch.cuda.memory_stats()
    assert free_after == free_before
    for key in ("allocation.all.allocated", "segment.all.allocated", "reserved_bytes.all.current"):
        assert stats_after.get(key) == stats_before.get(key), key
    assert torch.equal(out, ref)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    w = synthetic.WORKLOADS["flux_1024_4608"]          # 24 heads x 4608 tokens > 32768
    cfg = fa.make_config(w.batch, w.heads, w.tokens)
    x = torch.empty((1, 8, 1, 128), dtype=torch.bfloat16, device="cuda")
    wt = torch.ones(128, device="cuda")
    with pytest.raises(fa.FluxAttnError) as e:
        fa.flux_attn_forward_noalloc(cfg, x, x, x, *_geom(w), None, wt, wt, torch.empty_like(x))
    assert e.value.status == fa.FLUX_ATTN_ERR_INVALID_ARG
    assert "allocation-free limit" in str(e.value)
    fp8 = fa.make_config(1, 1, 8, precision=fa.FLUX_ATTN_FP8_E4M3)
    with pytest.raises(fa.FluxAttnError) as e:
        fa.flux_attn_forward_noalloc(fp8, x, x, x, 8, 0, 0, 0, 0, None, wt, wt, torch.empty_like(x))
    assert e.value.status == fa.FLUX_ATTN_ERR_UNSUPPORTED
    unknown = fa.make_config(1, 1, 8, precision=7)     # flux_attn_create answers INVALID_ARG here too
    with pytest.raises(fa.FluxAttnError) as e:
        fa.flux_attn_forward_noalloc(unknown, x, x, x, 8, 0, 0, 0, 0, None, wt, wt, torch.empty_like(x))
    assert e.value.status == fa.FLUX_ATTN_ERR_INVALID_ARG
