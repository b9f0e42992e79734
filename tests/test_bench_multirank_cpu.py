"""The multi-rank logic of bench.py on CPU: two gloo ranks reduce their step
times to the slowest one and compute the same whole-job rate (weak scaling:
each rank runs the full per-rank workload, no data-path collective)."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [12.0, 15.0][rank]
    mx = bench.reduce_max(local_ms, dist)
    rate = bench.whole_job_rate(2.0e12, 10, world, mx)
    out[rank] = (mx, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_rank():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1]
    mx, rate = out[0]
    assert mx == 15.0
    # 2 ranks x 10 steps x 2 TFLOP in 15 ms
    assert rate == pytest.approx(2 * 10 * 2.0e12 / 15e-3)


def test_single_process_needs_no_group():
    import bench
    assert bench.reduce_max(3.5) == 3.5
    assert bench.whole_job_rate(1.0, 4, 1, 2.0) == pytest.approx(2000.0)
