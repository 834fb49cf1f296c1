"""The benchmark's multi-rank host logic on CPU: two gloo ranks.

With N > 1 GPUs every rank runs an independent replica of the workload (the
path has no cross-GPU step on this hardware), and the job's time is the MAX of
the ranks' times. These tests run that aggregation over a real two-process
gloo group, with per-rank times chosen so that each rank is slowest in one
of the two measurements.
"""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        step_ms = [5.0, 7.5][rank]   # rank 1 is slower per step
        e2e_ms = [9.0, 8.0][rank]    # rank 0 is slower end to end
        got = bench.max_over_ranks([step_ms, e2e_ms], torch.device("cpu"))
        value = bench.job_throughput(world, 8.8e12, got[0])
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{got[0]} {got[1]} {value}\n")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        step, e2e, value = map(float, open(tmp_path / f"rank{rank}.txt").read().split())
        assert step == 7.5 and e2e == 9.0
        # both ranks' work (2 x 8.8 TFLOP) over the slower rank's 7.5 ms
        assert value == pytest.approx(2 * 8.8e12 / 7.5e-3 / 1e12)


def test_job_throughput_single_rank():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.job_throughput(1, 8.8e12, 5.5) == pytest.approx(1600.0)
