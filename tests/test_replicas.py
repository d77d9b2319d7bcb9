"""bench.py's N-replica aggregation on CPU: world-size-2 gloo ranks (no GPU)."""
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
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank 0 is slower on the step, rank 1 on the end-to-end pass
        got = bench.max_over_ranks([1.0 + rank, 10.0 * (2 - rank), 3.0], world)
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 20.0, 3.0]


def test_replica_throughput_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    # two replicas of 100 units, slowest step 2 ms -> 200 units / 2 ms
    assert bench.replica_throughput(2, 100.0, 2.0) == pytest.approx(1e5)
    assert bench.replica_throughput(1, 100.0, 2.0) == pytest.approx(5e4)
