"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The block has no exchange step, so N GPUs run N independent replicas; the only
cross-rank logic is the barrier and the max-over-ranks timing that turns
per-rank times into the whole-job throughput.  These tests run it with the
gloo backend in two processes.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, seconds, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        agg = bench.aggregate(tokens_per_rank=1000, seconds_this_rank=seconds[rank], world=world)
        q.put((rank, agg))
    finally:
        dist.destroy_process_group()


def test_aggregate_takes_slowest_rank_and_sums_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    seconds = [0.5, 2.0]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, seconds, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        assert res[r]["seconds"] == pytest.approx(2.0)
        assert res[r]["value"] == pytest.approx(2 * 1000 / 2.0)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    agg = bench.aggregate(500, 0.25, 1)
    assert agg["seconds"] == 0.25 and agg["value"] == 2000.0
