"""The bench's multi-GPU plumbing (one process per rank, weak scaling, no data-path
collective: only the barrier and the max over ranks of the timed region), run as two gloo
ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    # each rank's own time; every rank must see the maximum
    mine = 10.0 + 7.5 * rank
    results[rank] = bench.max_over_ranks(mine, w, torch.device("cpu"))
    bench.barrier(w)
    torch.distributed.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_max_time():
    world, port = 2, _free_port()
    manager = mp.get_context("spawn").Manager()
    results = manager.dict()
    mp.start_processes(_rank_main, args=(world, port, results), nprocs=world, join=True,
                       start_method="spawn")
    assert dict(results) == {0: 17.5, 1: 17.5}


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.25, 1, torch.device("cpu")) == 3.25
    bench.barrier(1)   # a no-op without a process group
