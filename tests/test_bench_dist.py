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


def test_topk_algorithmic_bytes_count_rows_longer_than_k():
    """The top-k line's byte count: rows longer than k read their logits,
    every row reads its length and writes k indices."""
    import bench
    rl = torch.tensor([1, 5, 8, 9, 100], dtype=torch.int32)
    assert bench.rows_bytes(rl, 8) == 4 * (9 + 100) + 4 * 5 + 4 * 5 * 8
    n = torch.arange(1, 8193, dtype=torch.int64)
    assert bench.rows_bytes(n.to(torch.int32), 2048) == (
        4 * int(n[n > 2048].sum()) + 4 * 8192 + 4 * 8192 * 2048)


def test_topk_reference_arm_prints_its_line():
    """bench.py --impl reference on the 8192-row top-k workload runs the
    oracle on host cores and prints one JSON line of the contract."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--workload", "topk_s8k_k2048", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
