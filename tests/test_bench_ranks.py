"""The multi-GPU bench path on CPU: two gloo ranks agree on the slowest rank's time and the
whole-job rate sums the ranks' work over it (replicas, no collective on the data path)."""
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


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    my_ms = [120.0, 150.0][rank]  # rank 1 is the slowest
    slowest = bench.max_over_ranks(my_ms, world, device="cpu")
    results[rank] = (slowest, bench.whole_job_rate(2.0e12, 10, slowest, world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    mgr = mp.Manager()
    results = mgr.dict()
    mp.spawn(_worker, args=(2, _free_port(), results), nprocs=2, join=True)
    assert results[0][0] == results[1][0] == 150.0
    # 2 ranks x 2e12 FLOP x 10 steps over 0.15 s
    assert results[0][1] == pytest.approx(2 * 2.0e12 * 10 / 0.150)


def test_single_process_is_its_own_max():
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(1.0e9, 4, 2.0, 1) == pytest.approx(2.0e12)
