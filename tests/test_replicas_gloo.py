"""The multi-rank path of bench.py on CPU: two gloo ranks (no GPU).

bench.py runs one independent replica per rank; the only cross-rank steps
are the barriers around the timed region, the max over ranks of the step
time and the whole-job rate.  These are checked here with real processes.
"""

import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, wsz, local = bench.rank_info()
        bench.barrier(dist)
        slowest = bench.max_over_ranks(10.0 + 5.0 * r, dist)
        seed = bench.replica_seed(1002, r)
        rate = bench.whole_job_rate(274.9e9, wsz, 1e-3)
        bench.barrier(dist)
        out[rank] = (r, wsz, local, slowest, seed, rate)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for rank, (r, wsz, local, slowest, seed, rate) in res.items():
        assert (r, wsz, local) == (rank, 2, rank)
        assert slowest == 15.0                      # the max over both ranks
        assert rate == pytest.approx(2 * 274.9e12)  # whole-job rate
    assert res[0][4] != res[1][4]                   # distinct replica seeds


def test_single_process_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    sys.path.insert(0, ROOT)
    import bench

    assert bench.rank_info() == (0, 1, 0)
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0
