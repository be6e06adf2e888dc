"""Multi-process host logic of the replica benchmark on CPU (gloo, 2 ranks):
the max-over-ranks step time and the summed whole-job work that bench.py
reports when N GPUs each run an independent replica."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.0][rank]           # per-rank step time
    work = [100.0, 100.0][rank]     # per-rank bytes per step (weak scaling: fixed per GPU)
    t = bench._max_over_ranks(dist, ms, torch.device("cpu"))
    w = bench._sum_over_ranks(dist, work, torch.device("cpu"))
    bench._barrier(dist)
    q.put((rank, t, w))
    dist.destroy_process_group()


def test_replica_aggregation_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 5.0, 200.0), (1, 5.0, 200.0)]


def test_single_process_is_identity():
    import bench
    assert bench._max_over_ranks(None, 2.5, torch.device("cpu")) == 2.5
    assert bench._sum_over_ranks(None, 7.0, torch.device("cpu")) == 7.0
    if not torch.cuda.is_available():
        pytest.skip("no GPU here: the bench body itself runs under -m gpu paths")
