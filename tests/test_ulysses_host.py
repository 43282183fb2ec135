"""Ulysses sequence parallelism on the host: two gloo ranks on the CPU (no GPU).

"Speed up image generation with FLUX 3 Image Klein on NVIDIA Blackwell GPUs",
section "Multi-GPU inference" (ulysses_size, cfg_size): the sequence is split
over the ranks of a group and an all-to-all turns it into a head split around
the attention.  Here each of two ranks holds half of the joint sequence; the
per-rank attention is the fp64 oracle on the rank's heads (the GPU path puts
flux_attn_forward there), and the reassembled chunks must equal the oracle on
the whole problem -- which checks the partition and both exchanges: a wrong
head group, token chunk or permutation moves rows between heads or tokens.
A second run checks the layout transforms alone, bit for bit, with a
position-coded tensor.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def _worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        import synthetic
        from diffusion_transformer_joint_txt_b300 import ulysses
        # layout transforms alone: element (b, n, h, d) carries its own coordinates
        B, N, H, D = 2, 8, 4, 128
        code = (np.arange(B)[:, None, None, None] * 1e6 + np.arange(N)[None, :, None, None] * 1e3
                + np.arange(H)[None, None, :, None] * 10 + (np.arange(D) % 7)[None, None, None, :])
        full = torch.from_numpy(code.astype(np.float32)).to(torch.bfloat16)
        chunk = full[:, rank * N // world:(rank + 1) * N // world].contiguous()
        heads = ulysses.seq_to_heads(chunk, world, None, dist)
        hp = H // world
        assert torch.equal(heads, full[:, :, rank * hp:(rank + 1) * hp])
        back = ulysses.heads_to_seq(heads, world, None, dist)
        assert torch.equal(back, chunk)
        # the attention through the exchange, against the oracle on the whole problem
        w = synthetic.Workload("ulysses", 2, 4, 8, 5, 6, 2, 3)          # N = 8 + 30 + 6 = 44
        inp = synthetic.make_inputs(w, seed=12)
        n = w.tokens

        def oracle_attend(q, k, v, txt, ih, iw, rh, rw, wq, wk, pos):
            bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
            o = oracle.attention_rows(bits(q), bits(k), bits(v), inp.pos, inp.w_q, inp.w_k, nthreads=1)
            return torch.from_numpy(o.astype(np.float32)).to(torch.bfloat16)

        ua = ulysses.UlyssesAttention(w.batch, w.heads, n, attend=oracle_attend)
        lo, hi = rank * n // world, (rank + 1) * n // world
        q, k, v = (_bf16(t)[:, lo:hi].contiguous() for t in (inp.q, inp.k, inp.v))
        out = ua.forward(q, k, v, w.txt_len, w.img_h, w.img_w, w.ref_h, w.ref_w)
        np.save(os.path.join(out_dir, "out%d.npy" % rank), out.float().numpy())
    finally:
        dist.destroy_process_group()


def test_ulysses_two_ranks_match_the_whole_problem(tmp_path):
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    import synthetic
    oracle.build()
    mp.spawn(_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    w = synthetic.Workload("ulysses", 2, 4, 8, 5, 6, 2, 3)
    inp = synthetic.make_inputs(w, seed=12)
    want = oracle.attention_rows(inp.q, inp.k, inp.v, inp.pos, inp.w_q, inp.w_k)
    got = np.concatenate([np.load(tmp_path / ("out%d.npy" % r)) for r in range(2)], axis=1)
    assert got.shape == want.shape
    # the ranks computed their heads in fp64 and returned bf16: bf16 rounding only
    np.testing.assert_allclose(got, want, rtol=2 ** -8, atol=1e-6)


def test_ulysses_rejects_shapes_it_cannot_split():
    import sys
    sys.path.insert(0, ROOT)
    from diffusion_transformer_joint_txt_b300 import ulysses

    class FakeDist:
        @staticmethod
        def get_world_size(group=None):
            return 4

        @staticmethod
        def get_rank(group=None):
            return 0

    orig = dist.get_world_size, dist.get_rank
    dist.get_world_size, dist.get_rank = FakeDist.get_world_size, FakeDist.get_rank
    try:
        with pytest.raises(ValueError):
            ulysses.UlyssesAttention(1, 6, 64, attend=lambda *a: None)          # 6 heads over 4 ranks
        ua = ulysses.UlyssesAttention(1, 8, 64, attend=lambda *a: None)
        x = torch.zeros((1, 10, 8, 128), dtype=torch.bfloat16)
        with pytest.raises(ValueError):
            ua.forward(x, x, x, 10, 3, 10)                                   # N = 40: fine count, wrong chunk
        with pytest.raises(ValueError):
            ua.forward(x, x, x, 2, 3, 11)                                    # N = 35 over 4 ranks
    finally:
        dist.get_world_size, dist.get_rank = orig
