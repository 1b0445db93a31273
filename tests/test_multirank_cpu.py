"""The multi-rank bench path on CPU: two gloo ranks, each timing its own
replica, must report the slowest rank's time and the whole job's tokens."""
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


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        e2e_ms = 12.0 + 1.0 * (1 - rank)  # rank 0 is slow end to end
        out = bench.aggregate_ranks(ms, e2e_ms, tokens_per_step=512, steps=4, world=world,
                                    device="cpu")
        results[rank] = out
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_takes_the_slowest_rank():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, results), nprocs=2, join=True,
                       start_method="spawn")
    for rank in (0, 1):
        ms, e2e_ms, tokens, value = results[rank]
        assert ms == 15.0 and e2e_ms == 13.0
        assert tokens == 512 * 4 * 2
        assert value == pytest.approx(tokens / 0.015)


def test_single_rank_aggregation_is_local():
    import bench
    ms, e2e_ms, tokens, value = bench.aggregate_ranks(8.0, 9.0, 100, 3, 1, "cpu")
    assert (ms, e2e_ms, tokens) == (8.0, 9.0, 300)
    assert value == pytest.approx(300 / 0.008)
