"""Multi-rank host logic of bench.py on CPU: two gloo ranks.

The bench runs one independent replica of the decode step per GPU (no
collective on the data path); the only cross-rank steps are the barrier
around the timed region and the maximum of the ranks' durations, which sets
the whole-job throughput.  Both run here over gloo, world size 2.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, _ = bench.dist_info()
        assert (w, r) == (world, rank)
        dist.barrier()
        mine = [10.0, 12.5][rank]   # rank 1 is the slower one
        got = bench.reduce_max_ms(mine, world, torch.device("cpu"))
        value = bench.whole_job_value(world, 256, 100, got)
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{got} {value}\n")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn",
                       join=True)
    for rank in range(world):
        got, value = map(float, open(tmp_path / f"r{rank}.txt").read().split())
        assert got == 12.5
        # 2 replicas x 256 queries x 100 steps in 12.5 ms
        assert value == pytest.approx(2 * 256 * 100 / 12.5e-3)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.reduce_max_ms(3.25, 1, torch.device("cpu")) == 3.25
    assert bench.whole_job_value(1, 256, 10, 2.0) == pytest.approx(256 * 10 / 2e-3)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import argparse

    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(steps=1, warmup=3, cpu_seconds=0.1)
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""
