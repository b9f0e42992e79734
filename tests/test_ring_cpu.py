"""The ring exchange on CPU ranks (gloo): every rank holds one block of Q, K
and V; at step t rank I must hold KV block (I - t) mod N, received intact
from rank I - 1, and the merged result must be the attention over the whole
sequence.  The device operations are replaced by the float64 oracle
(rotation, attention of one block with positions, merge of partials), so the
test checks the exchange schedule, the payloads and the merge order; the
same driver runs the library's kernels on GPUs."""

import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from yarn_rope_scaling_ntk_b300 import api, ring

S_BLOCK, B, HQ, HKV, D = 24, 1, 4, 2, 16
CFG = dict(kind="yarn", head_dim=D, theta_base=1e4, L_train=32, s=4.0)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(world):
    g = torch.Generator().manual_seed(9000 + world)
    S = S_BLOCK * world
    q = torch.randn(B, HQ, S, D, generator=g, dtype=torch.float64)
    k = torch.randn(B, HKV, S, D, generator=g, dtype=torch.float64)
    v = torch.randn(B, HKV, S, D, generator=g, dtype=torch.float64)
    return q, k, v


def oracle_ops(log):
    import oracle.attention as A
    import oracle.rope as R
    th, _, _ = R.inv_freq(CFG["kind"], D, CFG["theta_base"], CFG["L_train"], 0, CFG["s"])

    def rotate(cfg, x, pos0):
        pos = np.arange(pos0, pos0 + x.shape[2])
        return torch.from_numpy(R.rotate(x.numpy(), pos, th))

    def block(q, k, v, q_pos0, k_pos0, mask, sink, window, scale, out_dtype):
        log.append((k_pos0, k.clone(), v.clone()))
        G = q.shape[1] // k.shape[1]
        qp = np.arange(q_pos0, q_pos0 + q.shape[2])
        kp = np.arange(k_pos0, k_pos0 + k.shape[2])
        o = torch.zeros(q.shape, dtype=torch.float64)
        lse = torch.zeros(q.shape[:3], dtype=torch.float64)
        for b in range(q.shape[0]):
            for h in range(q.shape[1]):
                oo, ll = A.attention_rows(q[b, h].numpy(), qp, k[b, h // G].numpy(), v[b, h // G].numpy(), mask, sink,
                                          window, scale, k_pos=kp)
                o[b, h], lse[b, h] = torch.from_numpy(oo), torch.from_numpy(ll)
        return o, lse

    def merge(o_acc, lse_acc, o_part, lse_part, out):
        for b in range(o_acc.shape[0]):
            for h in range(o_acc.shape[1]):
                o, l = A.merge_partials([(o_acc[b, h].numpy(), lse_acc[b, h].numpy()),
                                         (o_part[b, h].numpy(), lse_part[b, h].numpy())])
                o_acc[b, h], lse_acc[b, h] = torch.from_numpy(o), torch.from_numpy(l)
        if out is not None:
            out.copy_(o_acc)

    return ring.RingOps(rotate, block, merge)


def _rank_main(rank, world, port, mask, sink, window, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q, k, v = _inputs(world)
        blk = slice(rank * S_BLOCK, (rank + 1) * S_BLOCK)
        log = []
        o, lse = ring.ring_attention(api.RopeConfig(**CFG), q[:, :, blk], k[:, :, blk].contiguous(),
                                     v[:, :, blk].contiguous(), mask=mask, sink=sink, window=window,
                                     ops=oracle_ops(log))
        out[rank] = (o.numpy(), lse.numpy(), [(kp, kk.numpy(), vv.numpy()) for kp, kk, vv in log])
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,mask,sink,window", [(2, "causal", 0, 0), (4, "causal", 0, 0),
                                                    (4, "sink_window", 2, 30), (3, "none", 0, 0)])
def test_ring_exchange_on_gloo_ranks(world, mask, sink, window):
    import oracle.attention as A
    import oracle.rope as R
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, mask, sink, window, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    q, k, v = _inputs(world)
    S = S_BLOCK * world
    th, _, ms = R.inv_freq(CFG["kind"], D, CFG["theta_base"], CFG["L_train"], 0, CFG["s"])
    scale = A.softmax_scale("yarn", CFG["s"], D)
    kr = R.rotate(k.numpy(), np.arange(S), th)
    for rank in range(world):
        o, lse, log = out[rank]
        # the blocks this rank computed, in ring order, each received intact
        want_order = A.ring_block_order(rank, world, mask)
        assert [kp // S_BLOCK for kp, _, _ in log] == want_order
        for kp, kk, vv in log:
            j = kp // S_BLOCK
            blk = slice(j * S_BLOCK, (j + 1) * S_BLOCK)
            assert np.array_equal(kk, kr[:, :, blk]), f"rank {rank}: K block {j} changed in transit"
            assert np.array_equal(vv, v[:, :, blk].numpy()), f"rank {rank}: V block {j} changed in transit"
        # the merged result is attention over the whole sequence
        rows = np.arange(rank * S_BLOCK, (rank + 1) * S_BLOCK)
        for h in range(HQ):
            qr = R.rotate(q[0, h, rows].numpy(), rows, th)
            want_o, want_l = A.attention_rows(qr, rows, kr[0, h // (HQ // HKV)], v[0, h // (HQ // HKV)].numpy(),
                                              mask, sink, window, scale)
            np.testing.assert_allclose(o[0, h], want_o, atol=1e-12)
            np.testing.assert_allclose(lse[0, h], want_l, atol=1e-12)


def test_ring_schedule_helpers():
    import oracle.attention as A
    for world in (1, 2, 5, 8):
        for rank in range(world):
            held = [ring.held_block(rank, t, world) for t in range(world)]
            assert sorted(held) == list(range(world))  # every block once
            for mask in ("causal", "none"):
                vis = [j for j in held if ring.block_visible(rank, j, mask)]
                assert vis == A.ring_block_order(rank, world, mask)
