"""The bench's multi-process path on CPU: two gloo ranks (replicas, no data-path
collective).  Checks the barrier, the max-over-ranks of the elapsed time, the
whole-job aggregation of tokens/s and that the reference arm runs on rank 0 only."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.Dist()
    try:
        dist.barrier()
        elapsed = [10.0, 25.0][rank]  # this rank's timed region, ms
        m = dist.max(elapsed)
        T, steps = 128, 4
        value = dist.world * T * steps / (m / 1e3)
        args = type("A", (), {"steps": 1, "warmup": 0})()
        ref = bench.run_reference(args, dist, None) if rank != 0 else "rank0"
        out.put((rank, dist.world, m, value, ref))
    finally:
        dist.close()


def test_two_gloo_ranks_take_the_max_and_aggregate():
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
    for rank, world, m, value, ref in res:
        assert world == 2
        assert m == 25.0  # both ranks see the slowest rank's time
        assert value == pytest.approx(2 * 128 * 4 / 0.025)
    assert res[1][4] is None  # rank 1 does no reference work and prints nothing
