"""Host logic of the multi-GPU path (replicas only), on CPU with two gloo ranks: the job
time is the slowest rank's and the job throughput counts every rank's tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank: int, world: int, port: int, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r timed (10 + r) ms for 100 steps and (20 + 2 r) ms for 10 end-to-end steps
    res = bench.combine_ranks(10.0 + rank, 20.0 + 2 * rank, 100, 10, world)
    out[rank] = res
    dist.barrier()
    dist.destroy_process_group()


def test_combine_ranks_takes_the_slowest_rank_and_counts_all_tokens():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        got = dict(out)
    for rank in range(world):
        ms, e2e_ms, tok_s, e2e_tok_s = got[rank]
        assert ms == 11.0 and e2e_ms == 22.0
        assert tok_s == pytest.approx(2 * 100 / 0.011)
        assert e2e_tok_s == pytest.approx(2 * 10 / 0.022)


def test_combine_ranks_single_process():
    import bench
    ms, e2e_ms, tok_s, e2e_tok_s = bench.combine_ranks(4.0, 8.0, 40, 4, 1)
    assert (ms, e2e_ms) == (4.0, 8.0)
    assert tok_s == pytest.approx(10000.0) and e2e_tok_s == pytest.approx(500.0)
