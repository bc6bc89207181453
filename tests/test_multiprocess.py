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


def _host_path_rank(rank, world, port, results):
    """One rank's host half of the path: its own prompts packed by the library's FFD packer, the
    packed stream's metadata, and a host-built attention plan for its batch; checked against the
    oracle's packer, then gathered so the test can compare ranks."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import scheduling as osched
        from sparsified_long_context_gb300 import binding as B
        rng = np.random.default_rng(100 + rank)
        lengths = rng.integers(1, 900, 24).astype(np.int32)
        order, bin_cu = B.unip_ffd_pack(lengths, 1024)
        ref_order, ref_bin_cu = osched.ffd_order(lengths, 1024)
        assert np.array_equal(order, ref_order) and np.array_equal(bin_cu, ref_bin_cu)
        cu, pos, src = B.unip_pack_metadata(lengths, order)
        rcu, rpos, rsrc = osched.pack_metadata(lengths, order)
        assert np.array_equal(cu, rcu) and np.array_equal(pos, rpos) and np.array_equal(src, rsrc)
        # the rank's packed stream as one attention call: one segment per prompt, in packed order
        plan = B.AttentionPlan(cu, None, num_heads_q=8, num_heads_kv=2, head_dim=64, page_size=0,
                               max_pages_per_seq=0, num_sms=152)
        info = plan.info
        plan.close()
        gathered = [None] * world
        dist.all_gather_object(gathered, (rank, lengths.tolist(), int(cu[-1]), info["items"], info["host"]))
        results[rank] = gathered
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_run_the_host_path_on_their_own_batches():
    world, port = 2, _free_port()
    mgr = mp.Manager()
    results = mgr.dict()
    mp.spawn(_host_path_rank, args=(world, port, results), nprocs=world, join=True)
    g0, g1 = results[0], results[1]
    assert g0 == g1                                          # every rank sees every rank's summary
    (r0, len0, n0, items0, host0), (r1, len1, n1, items1, host1) = g0
    assert (r0, r1) == (0, 1) and len0 != len1              # independent batches, no shared data
    assert n0 == sum(len0) and n1 == sum(len1)              # every token of a rank's prompts is packed
    assert host0 and host1 and items0 > 0 and items1 > 0   # both plans built on the host
