"""Ulysses sequence parallelism around the joint attention (host side).

"Speed up image generation with FLUX 3 Image Klein on NVIDIA Blackwell GPUs",
section "Multi-GPU inference": the runtime splits each classifier-free-guidance
branch's sequence over a group of GPUs (Ulysses, ulysses_size 4 with cfg_size 2
on eight GPUs) and handles the sequence split, the distributed attention and
the output gather.  Ulysses turns the sequence split into a head split around
the attention:

  rank r of a group of P holds tokens [r N/P, (r+1) N/P) of q, k, v with all H
  heads; an all-to-all gives it all N tokens of heads [r H/P, (r+1) H/P); the
  attention of those heads runs whole on the rank (flux_attn_forward: the
  QK-norm + RoPE prologue and the joint attention, which need every token of a
  head); a second all-to-all returns each rank's token chunk with all heads.

Layout per rank: q, k, v, out bf16 [B, N/P, H, 128]; the token order of the
joint sequence is the usual [text | image | reference], cut into P equal
contiguous chunks.  N and H must be multiples of P.  Positions come from the
geometry (or an explicit [N, 3] pos_ids on every rank), so the exchange moves
only q, k, v and the output.

Two exchanges of 3 + 1 tensors per call, B N H 128 bf16 each, of which each
rank sends (P - 1) / P.  Classifier-free-guidance parallelism (cfg_size) is
plain data parallelism over the batch: give each CFG group its own process
group and its own batch rows; no exchange crosses groups.

The exchange is torch.distributed.all_to_all_single on the given process
group (NCCL between GPUs; gloo on the CPU for the multi-process tests), with
bf16 data carried as int32 pairs (head_dim 128 is even) so that any backend
moves the bits unchanged.  The per-rank attention defaults to the C ABI's
flux_attn_forward on the rank's device; no step of it runs on the host.
"""
from __future__ import annotations

from typing import Callable, Optional

HEAD_DIM = 128


def _a2a(x, group, dist):
    """all_to_all_single of a [P, ...] tensor: chunk p goes to rank p, and
    chunk p of the result came from rank p; bf16 travels as int32 pairs."""
    import torch
    send = x.contiguous()
    if send.element_size() == 2:
        send = send.view(torch.int32)
    recv = torch.empty_like(send)
    dist.all_to_all_single(recv, send, group=group)
    return recv.view(x.dtype) if x.element_size() == 2 else recv


def seq_to_heads(x, world: int, group, dist):
    """[B, N/P, H, D] sequence chunk -> [B, N, H/P, D] head group of this rank."""
    B, n_loc, H, D = x.shape
    hp = H // world
    send = x.reshape(B, n_loc, world, hp, D).permute(2, 0, 1, 3, 4)       # [P(head group), B, n, hp, D]
    recv = _a2a(send, group, dist)                                          # [P(token chunk), B, n, hp, D]
    return recv.permute(1, 0, 2, 3, 4).reshape(B, world * n_loc, hp, D)


def heads_to_seq(y, world: int, group, dist):
    """[B, N, H/P, D] head group -> [B, N/P, H, D] sequence chunk of this rank."""
    B, N, hp, D = y.shape
    n_loc = N // world
    send = y.reshape(B, world, n_loc, hp, D).permute(1, 0, 2, 3, 4)        # [P(token chunk), B, n, hp, D]
    recv = _a2a(send, group, dist)                                          # [P(head group), B, n, hp, D]
    return recv.permute(1, 2, 0, 3, 4).reshape(B, n_loc, world * hp, D)


class UlyssesAttention:
    """Joint attention over a sequence split across the ranks of `group`.

    attend(q, k, v, geometry, q_norm_w, k_norm_w, pos_ids) is the attention of
    the rank's heads over all N tokens, [B, N, H/P, 128] in and out; by default
    a FluxAttention handle of B batch rows and H/P heads on the current device
    (precision and the handle's other settings from **handle_kw).
    """

    def __init__(self, batch: int, num_heads: int, max_tokens: int, group=None,
                 attend: Optional[Callable] = None, **handle_kw):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        if num_heads % self.world:
            raise ValueError("num_heads = %d is not a multiple of the group size %d" % (num_heads, self.world))
        self.batch, self.num_heads, self.max_tokens = batch, num_heads, max_tokens
        self.local_heads = num_heads // self.world
        self._attn = None
        if attend is None:
            from . import FluxAttention
            self._attn = FluxAttention(batch, self.local_heads, max_tokens, **handle_kw)
            attend = self._flux_attend
        self.attend = attend

    def _flux_attend(self, q, k, v, txt_len, img_h, img_w, ref_h, ref_w, q_norm_w, k_norm_w, pos_ids):
        return self._attn.forward(q, k, v, txt_len, img_h, img_w, ref_h, ref_w, q_norm_w, k_norm_w, pos_ids)

    def close(self):
        if self._attn is not None:
            self._attn.close()
            self._attn = None

    def forward(self, q, k, v, txt_len: int, img_h: int, img_w: int, ref_h: int = 0, ref_w: int = 0,
                q_norm_w=None, k_norm_w=None, pos_ids=None):
        """q, k, v: this rank's sequence chunk, bf16 [B, N/P, H, 128]; returns
        the attention output of the same chunk, bf16 [B, N/P, H, 128]."""
        n = txt_len + img_h * img_w + ref_h * ref_w
        if n % self.world:
            raise ValueError("N = %d tokens is not a multiple of the group size %d" % (n, self.world))
        shape = (self.batch, n // self.world, self.num_heads, HEAD_DIM)
        for t, name in ((q, "q"), (k, "k"), (v, "v")):
            if tuple(t.shape) != shape:
                raise ValueError("%s must be [B, N/P, H, 128] = %s, got %s" % (name, shape, tuple(t.shape)))
        qh, kh, vh = (seq_to_heads(t, self.world, self.group, self.dist) for t in (q, k, v))
        oh = self.attend(qh, kh, vh, txt_len, img_h, img_w, ref_h, ref_w, q_norm_w, k_norm_w, pos_ids)
        return heads_to_seq(oh, self.world, self.group, self.dist)
