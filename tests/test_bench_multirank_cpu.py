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


def _bench_lines(*args, env=None):
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), *args], capture_output=True, text=True,
                       timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]


@pytest.mark.parametrize("n", [2, 4])
def test_bench_gpus_n_starts_n_ranks_itself(n):
    """``bench.py --gpus N`` with no launcher environment starts N rank
    processes that form one group; rank 0 alone prints one line for the job."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    lines = _bench_lines("--gpus", str(n), "--steps", "2", "--launcher-check", env=env)
    assert len(lines) == 1
    assert lines[0]["n_gpus"] == n and lines[0]["ranks_joined"] == n


def test_bench_under_a_launcher_does_not_start_ranks_again():
    """Under torchrun (WORLD_SIZE set) each process is one rank already: a
    single-rank environment runs one process and prints one line."""
    env = dict(os.environ, RANK="0", LOCAL_RANK="0", WORLD_SIZE="1")
    lines = _bench_lines("--gpus", "2", "--steps", "2", "--launcher-check", env=env)
    assert len(lines) == 1 and lines[0]["n_gpus"] == 1


@pytest.mark.parametrize("n", [2, 4])
def test_bench_ring_mode_starts_n_ranks_and_hands_each_the_ring_order(n):
    """``bench.py --ring --gpus N``: N ranks pass their KV blocks around the
    ring (gloo point-to-point on the CPU here) and each rank is handed, at
    step t, block (rank - t) mod N, skipping future blocks."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    lines = _bench_lines("--ring", "--gpus", str(n), "--steps", "2", "--launcher-check", env=env)
    assert len(lines) == 1
    assert lines[0]["mode"] == "ring" and lines[0]["n_gpus"] == n and lines[0]["ring_order_ok"] is True


def test_reference_arm_line_matches_the_step_config():
    """``bench.py --impl reference`` (the float64 oracle on the host cores)
    prints one line with the same metric, unit and config as the GPU arm."""
    import bench
    from yarn_rope_scaling_ntk_b300 import workloads as W
    lines = _bench_lines("--impl", "reference", "--steps", "1", "--warmup", "0")
    assert len(lines) == 1
    ln = lines[0]
    assert ln["impl"] == "reference" and ln["metric"] == bench.METRIC and ln["unit"] == "TFLOP/s"
    assert ln["config"] == bench.step_config(W.LLAMA2_7B, 1)
    assert ln["value"] > 0 and ln["ms_per_step"] > 0 and ln["cpu_baseline"]["kind"] == "oracle"
    assert ln["e2e"]["h2d_bytes_per_step"] == 0 and ln["e2e"]["d2h_bytes_per_step"] == 0
