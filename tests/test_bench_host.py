"""Host-side logic of bench.py: the replica aggregation over ranks (gloo,
world size 2, on CPU) and the clock-record parser."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.init_dist(world, "gloo")
    my_seconds = 1.0 + rank            # rank 1 is the slow one
    bench.barrier(world)
    slowest = bench.max_over_ranks(my_seconds, world)
    value = bench.whole_job_gbps(4e9, 10, world, slowest)
    results[rank] = (slowest, value)
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_count_every_rank():
    world = 2
    manager = mp.Manager()
    results = manager.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        slowest, value = results[r]
        assert slowest == 2.0
        # 2 ranks x 10 steps x 4 GB over the slowest rank's 2 s
        assert value == pytest.approx(2 * 10 * 4e9 / 2.0 / 1e9)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)


def test_clock_parser_median_and_reasons():
    lines = [
        "0, GPU-abc, 1900, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n",
        "0, GPU-abc, 1950, 2070, 1000.0, 0x4, Not Active, Not Active, Not Active, Active\n",
        "0, GPU-abc, 2000, 2070, 1100.0, 0x0, Not Active, Not Active, Not Active, Not Active\n",
        "1, GPU-other, 300, 2070, 100.0, 0x0, Active, Not Active, Not Active, Not Active\n",
        "garbage\n",
    ]
    got = bench.parse_clock_csv(lines, "GPU-abc")
    assert got == {"sm_mhz": 1950.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert bench.parse_clock_csv([], None) is None
