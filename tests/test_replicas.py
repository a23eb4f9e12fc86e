"""bench.py's replica mode on CPU: two gloo ranks, each with its own step time;
the aggregate takes the slowest rank's time and counts both ranks' bytes."""
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


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, _ = bench.dist_env()
    dist = bench.dist_init(w, "gloo")
    ms = 2.0 if r == 0 else 3.0          # rank 1 is slower
    agg_ms, value = bench.aggregate(ms, 0.5, w)   # 0.5 GB per step per rank
    q.put((r, agg_ms, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, agg_ms, value in res:
        assert agg_ms == pytest.approx(3.0)
        assert value == pytest.approx(2 * 0.5 / 3e-3)


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(2.0, 0.5, 1) == (2.0, pytest.approx(250.0))


def test_percentiles_of_step_times():
    sys.path.insert(0, ROOT)
    import bench
    xs = [float(v) for v in range(100, 0, -1)]   # 1 .. 100 ms, unsorted
    p = bench.pcts(xs)
    assert p == {"p10": 11.0, "p50": 51.0, "p90": 90.0}
    assert bench.pcts([7.0]) == {"p10": 7.0, "p50": 7.0, "p90": 7.0}
