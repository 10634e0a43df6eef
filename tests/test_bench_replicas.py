"""bench.py's multi-process plumbing on the CPU: two gloo ranks, barrier, max over ranks.

With N GPUs the benchmark runs N independent replicas (the collective path
does not shard across GPUs); the only cross-process steps are the barriers
around the timed region and the max of the ranks' times.  Those run here as
two CPU processes on the gloo backend.
"""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    d.init("gloo")
    d.barrier()
    got = d.max(float(10 + rank))
    d.barrier()
    d.close()
    q.put((rank, got, d.world))


def test_two_gloo_ranks_take_the_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(res) == [(0, 11.0, 2), (1, 11.0, 2)]


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    if d.world != 1:
        pytest.skip("running under a launcher")
    d.init("gloo")
    d.barrier()
    assert d.max(3.5) == 3.5
