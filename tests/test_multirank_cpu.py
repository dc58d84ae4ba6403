"""The N-GPU measurement path's host logic on two gloo ranks (CPU, no GPU).

With N ranks every rank processes its own copy of the workload (independent
units, no data-path collective); the whole-job value is the work of all ranks
divided by the slowest rank's time.  This runs bench.py's own reduction helpers
on world_size 2 and checks them against the same numbers computed in one process.
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


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from sliding_window_attention_swa_gb300 import inputs as I

        work = bench.prefill_flops(I.MISTRAL)          # each rank: one full workload
        seconds = 0.001 * (1.0 + 0.25 * rank)           # rank 1 is the slowest
        rate = bench.job_rate(work, seconds, world, torch.device("cpu"))
        slowest = bench.reduce_over_ranks(seconds, "max", world, torch.device("cpu"))
        results[rank] = (rate, slowest, work)
    finally:
        dist.destroy_process_group()


def test_two_rank_job_rate():
    world = 2
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), results), nprocs=world, start_method="spawn")
    assert set(results.keys()) == {0, 1}
    rate0, slow0, work = results[0]
    rate1, slow1, _ = results[1]
    assert slow0 == slow1 == pytest.approx(0.00125)
    assert rate0 == rate1 == pytest.approx(2 * work / 0.00125)
