"""Ring attention across ranks: the exchange step around the per-device calls.

A sequence of N * bs tokens is split into N contiguous blocks; rank I holds
query block I and key/value block I ("Context Window Scaling ...", Section 5:
each GPU owns one block of Q, K and V).  At step t rank I holds KV block
(I - t) mod N: it sends the block it holds to rank I + 1 and receives the next
one from rank I - 1 while it computes attention of its queries against the
block it holds (same section, Overlapping P2P Communication).  Blocks after I
hold future tokens and are skipped under a causal or sink-window mask (FAQ 2)
but still passed on.  The partial results are combined exactly by their
log-sum-exp ("Context Length Extension", Ring Attention: partial results
combined using online softmax).

Each rank rotates its own Q and K once, at their global positions, so a KV
block travels already rotated.  The per-block attention and the merge are the
library's ``attn_fwd_prefill_kv_block`` and ``attn_merge_partial``; the
exchange is ``torch.distributed`` point-to-point (NCCL on GPUs): both
transfers of a step are posted as one batch before the step's attention call
and waited for after it, into a second pair of buffers.  Received blocks
always land in this rank's own memory.

``RingRank`` is the per-rank computation and ``RingOps`` its three
operations (rotate, one block, merge); ``ring_attention`` drives one rank over
a process group and ``ring_attention_one_process`` drives all ranks in one
process (the exchange becomes a hand-over of tensors), which runs the same
per-rank computation on one GPU.
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Callable

import torch

from . import api


def held_block(rank: int, step: int, world: int) -> int:
    """KV block rank ``rank`` holds at step ``step``: it receives from rank - 1."""
    return (rank - step) % world


def block_visible(q_block: int, k_block: int, mask: str) -> bool:
    """Whether any query of block ``q_block`` can see a key of ``k_block``:
    every block at or before the query block under a causal or sink-window
    mask, every block without a mask."""
    return mask == "none" or k_block <= q_block


@dataclass
class RingOps:
    """The three device operations of a ring rank.

    rotate(cfg, x, pos0) -> x rotated at positions pos0 + s (same dtype).
    block(q, k, v, q_pos0, k_pos0, mask, sink, window, scale, out_dtype) ->
        (o, lse): attention of the (rotated) queries against one (rotated) KV
        block, o normalised over that block and lse its log-sum-exp.
    merge(o_acc, lse_acc, o_part, lse_part, out) -> None: merge a partial
        into the float32 accumulator in place; ``out`` (or None) receives the
        merged O as well, in its own dtype.
    """
    rotate: Callable
    block: Callable
    merge: Callable


def cuda_ops(stream=None) -> RingOps:
    """The library's kernels (the product path)."""

    def rotate(cfg, x, pos0):
        return api.rope_apply(cfg, x, pos0=pos0, stream=stream)

    def block(q, k, v, q_pos0, k_pos0, mask, sink, window, scale, out_dtype):
        cfg = api.RopeConfig(kind="none", head_dim=q.shape[-1])
        return api.attn_fwd_prefill_kv_block(cfg, q, k, v, q_pos0, k_pos0, mask=mask, sink=sink, window=window,
                                             softmax_scale=scale, out_dtype=out_dtype, stream=stream)

    def merge(o_acc, lse_acc, o_part, lse_part, out):
        api.attn_merge_partial(o_acc, lse_acc, o_part, lse_part, out=out, stream=stream)

    return RingOps(rotate, block, merge)


class RingRank:
    """The computation of one rank of the ring.

    q [B, Hq, bs, d] and k, v [B, Hkv, bs, d] are block ``rank`` of the
    sequence (positions rank * bs ...).  ``compute(t, k_blk, v_blk)`` folds
    the KV block held at step t into the running result; ``result()``
    returns (o [B, Hq, bs, d] in q's dtype, lse [B, Hq, bs] float32)."""

    def __init__(self, cfg: api.RopeConfig, q, k, v, rank: int, world: int, mask: str = "causal", sink: int = 0,
                 window: int = 0, softmax_scale: float = 0.0, ops: RingOps | None = None):
        if mask not in ("causal", "sink_window", "none"):
            raise ValueError(f"unknown mask {mask!r}")
        if not 0 <= rank < world:
            raise ValueError("rank must lie in [0, world)")
        B, Hq, bs, d = q.shape
        if k.shape[0] != B or k.shape[2:] != (bs, d) or v.shape != k.shape:
            raise ValueError("k and v must be [B, Hkv, bs, d] with q's block size")
        self.ops = ops if ops is not None else cuda_ops()
        self.rank, self.world, self.bs = rank, world, bs
        self.mask, self.sink, self.window = mask, sink, window
        self.dtype = q.dtype
        pos0 = rank * bs
        if cfg.kind == "none":
            self.q, self.k = q, k
            ms = 1.0 if cfg.mscale_override <= 0 else cfg.mscale_override
        else:
            self.q = self.ops.rotate(cfg, q, pos0)
            self.k = self.ops.rotate(cfg, k, pos0)
            _, _, ms = api.yarn_inv_freq(cfg)
        self.v = v
        self.scale = softmax_scale if softmax_scale > 0 else ms * ms / math.sqrt(d)
        self.order = [held_block(rank, t, world) for t in range(world)]
        self.computed = [j for j in self.order if block_visible(rank, j, mask)]
        self.acc = self.lse = self.out = None

    def compute(self, step: int, k_blk, v_blk):
        j = self.order[step]
        if not block_visible(self.rank, j, self.mask):
            return
        only = len(self.computed) == 1
        last = j == self.computed[-1]
        # a single block is the result itself; otherwise float32 partials are
        # merged and the last merge writes the result in the input dtype
        o, lse = self.ops.block(self.q, k_blk, v_blk, self.rank * self.bs, j * self.bs, self.mask, self.sink,
                                self.window, self.scale, self.dtype if only else torch.float32)
        if self.acc is None:
            self.acc, self.lse = o, lse
            if only:
                self.out = o
            return
        if last and self.dtype != torch.float32:
            self.out = torch.empty(self.acc.shape, dtype=self.dtype, device=self.acc.device)
        self.ops.merge(self.acc, self.lse, o, lse, self.out if last else None)
        if last and self.out is None:
            self.out = self.acc

    def result(self):
        return self.out, self.lse


def ring_attention(cfg: api.RopeConfig, q, k, v, group=None, mask: str = "causal", sink: int = 0, window: int = 0,
                   softmax_scale: float = 0.0, ops: RingOps | None = None):
    """This rank's part of ring attention over ``group`` (default: the whole
    world): q, k, v are block ``rank`` of the sequence.  Returns (o, lse) for
    this rank's queries.  Every rank of the group must call it."""
    import torch.distributed as dist
    rank = dist.get_rank(group)
    world = dist.get_world_size(group)
    r = RingRank(cfg, q, k, v, rank, world, mask, sink, window, softmax_scale, ops)
    nxt_rank = dist.get_global_rank(group, (rank + 1) % world) if group is not None else (rank + 1) % world
    prv_rank = dist.get_global_rank(group, (rank - 1) % world) if group is not None else (rank - 1) % world
    cur_k, cur_v = r.k.contiguous(), r.v.contiguous()
    spare_k, spare_v = torch.empty_like(cur_k), torch.empty_like(cur_v)
    for t in range(world):
        works = []
        if t < world - 1:
            ops_ = [dist.P2POp(dist.isend, cur_k, nxt_rank, group), dist.P2POp(dist.isend, cur_v, nxt_rank, group),
                    dist.P2POp(dist.irecv, spare_k, prv_rank, group), dist.P2POp(dist.irecv, spare_v, prv_rank, group)]
            works = dist.batch_isend_irecv(ops_)
        r.compute(t, cur_k, cur_v)
        for w in works:
            w.wait()
        if t < world - 1:
            cur_k, spare_k = spare_k, cur_k
            cur_v, spare_v = spare_v, cur_v
    return r.result()


def ring_attention_one_process(cfg: api.RopeConfig, q_blocks, k_blocks, v_blocks, mask: str = "causal",
                               sink: int = 0, window: int = 0, softmax_scale: float = 0.0,
                               ops: RingOps | None = None):
    """Every rank of a ring of N = len(q_blocks) in this process, in lock
    step: at each step every rank computes on the block it holds, then each
    rank's block is handed to the next rank.  Returns [(o, lse)] per rank."""
    world = len(q_blocks)
    ranks = [RingRank(cfg, q_blocks[i], k_blocks[i], v_blocks[i], i, world, mask, sink, window, softmax_scale, ops)
             for i in range(world)]
    held = [(r.k, r.v) for r in ranks]
    for t in range(world):
        for i, r in enumerate(ranks):
            r.compute(t, *held[i])
        held = [held[(i - 1) % world] for i in range(world)]  # rank i receives from rank i - 1
    return [r.result() for r in ranks]
