"""The N > 1 bench path (replicas only: independent decode replicas, no
data-path collective) on CPU with two gloo ranks: the barrier, the
max-over-ranks timing and the whole-job per-call figure."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist = bench.init_dist(world, "gloo")
    bench.barrier(dist)
    mine = 10.0 + 5.0 * rank                    # rank 1 is the slow replica
    slowest = bench.reduce_max(mine, dist, "cpu")
    out[rank] = (slowest, bench.whole_job_us_per_call(slowest, 4, 78, world))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    assert out[0] == out[1]
    slowest, per_call = out[0]
    assert slowest == 15.0
    assert per_call == pytest.approx(15.0 * 1e3 / (4 * 78 * 2))


def test_single_replica_needs_no_process_group():
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.reduce_max(3.5, None) == 3.5
    assert bench.whole_job_us_per_call(2.0, 2, 10, 1) == 100.0
