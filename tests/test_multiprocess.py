"""The multi-rank bench path on CPU with the gloo backend (world size 2).

Segments are independent problems, so ranks run independent batches with no
collective on the data path; the only cross-rank operations are the barrier
around the timed region and the max over ranks of the elapsed time.
"""
import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, _ = bench.dist_setup(None)
        assert (w, r) == (world, rank)
        wl = bench.rank_seed_workload("tiny_packed", rank)
        dist.barrier()
        slowest = bench.max_over_ranks(10.0 + rank, dist)
        results[rank] = (slowest, int(wl.q[:8].astype(np.int64).sum()), float(bench.useful_attention_flops(wl)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_run_independent_batches_and_report_the_slowest():
    world, port = 2, _free_port()
    mgr = mp.Manager()
    results = mgr.dict()
    mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
    assert results[0][0] == results[1][0] == 11.0          # max over ranks
    assert results[0][1] != results[1][1]                  # different batches per rank
    assert results[0][2] == results[1][2]                  # same shape, same useful work per rank


def test_single_process_aggregation_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
