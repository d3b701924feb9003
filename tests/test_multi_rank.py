"""Multi-process aggregation of the benchmark, on CPU with the gloo backend.

The path has no exchange step (every (query, head) is independent), so N GPUs
run N independent replicas; the benchmark takes the slowest rank's time and
reports the whole job's throughput.  This runs that logic with two gloo ranks.
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 100.0 + 50.0 * rank          # rank 1 is the slow replica
    rate, total = bench.whole_job_rate(1e9, 10, local_ms, world, torch.device("cpu"))
    bench.barrier(world)
    out[rank] = (rate, total)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_replica():
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    # both ranks agree on the slowest time (150 ms) and on 2 replicas x 1e9 units x 10 steps
    for rank in (0, 1):
        rate, total = out[rank]
        assert total == pytest.approx(150.0)
        assert rate == pytest.approx(2 * 1e9 * 10 / 0.150)


def test_single_rank_is_identity():
    import bench
    rate, total = bench.whole_job_rate(5.0, 4, 2000.0, 1, torch.device("cpu"))
    assert total == 2000.0 and rate == pytest.approx(10.0)
