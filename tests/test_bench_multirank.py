"""The replicas path of bench.py on CPU: two gloo ranks, max-over-ranks timing and the
whole-job rate (every rank's units over the slowest rank's time)."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r pretends its timed loop took 10 + 5r ms and its end-to-end step 3 + r ms
    t, e = bench.slowest_rank(dist, [10.0 + 5 * rank, 3.0 + rank], torch.device("cpu"))
    rate = bench.whole_job_rate(world, 100.0, t * 1e-3)
    dist.barrier()
    out[rank] = (t, e, rate)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        t, e, rate = res[rank]
        assert t == 15.0 and e == 4.0
        assert rate == pytest.approx(2 * 100.0 / 0.015)


def test_single_process_without_group():
    import bench
    assert bench.slowest_rank(None, [1.5, 2.5], torch.device("cpu")) == [1.5, 2.5]
    assert bench.whole_job_rate(1, 10.0, 2.0) == 5.0
