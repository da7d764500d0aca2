"""The multi-rank bench path on CPU: two gloo ranks run the helpers bench.py
uses for N > 1 (max-over-ranks step time, whole-job throughput of replicas)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    w, r, _ = bench.dist_setup(world, backend="gloo")
    assert (w, r) == (world, rank)
    step_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    bench.barrier(w)
    t = bench.max_over_ranks(step_ms, w)
    out[rank] = (t, bench.job_throughput(1000.0, t, w))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        t, thr = res[rank]
        assert t == pytest.approx(15.0)
        assert thr == pytest.approx(world * 1000.0 / 15e-3)
