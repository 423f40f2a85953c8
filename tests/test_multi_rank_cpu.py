"""The N>1 path of bench.py on CPU: two gloo ranks run the same replica
workload description, take the max of their times and the sum of their work
(no data-path collective: the attention partitions into independent
requests), and agree on the whole-job number."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import workloads as wl
        # every rank builds the same replica workload (weak scaling)
        store = wl.cfg1_tiny("cpu")
        call = wl.whole_prefill(store)
        flops = bench.prefill_flops(call, 64, 4)
        local = [0.010 * (rank + 1), 0.002 * (world - rank)]  # fake per-rank seconds
        value, tmax = bench.aggregate_over_ranks(local, flops, steps=5, dist=dist)
        dist.barrier()
        out[rank] = (value, tmax, flops)
    finally:
        dist.destroy_process_group()


def test_two_replica_ranks_agree_on_the_whole_job_number():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
        assert p.exitcode == 0
    v0, t0, f0 = out[0]
    v1, t1, f1 = out[1]
    assert f0 == f1  # identical replicas
    assert t0 == t1 == [0.020, 0.004]  # max over ranks, item by item
    assert v0 == v1 == pytest.approx(world * f0 * 5 / 0.020)
