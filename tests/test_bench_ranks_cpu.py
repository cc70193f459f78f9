"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): every rank
joins the barrier, the reported throughput is the units all ranks processed
divided by the slowest rank's time (replicas, no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    import bench
    ranks = bench.Ranks(world)
    try:
        ranks.barrier()
        units = 1000.0 * (rank + 1)      # ranks process different amounts
        seconds = 0.5 + rank * 0.25       # rank 1 is the slowest
        value, slowest = bench.aggregate(units, seconds, ranks)
        q.put((rank, value, slowest))
    finally:
        ranks.close()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for _, value, slowest in got:
        assert slowest == pytest.approx(0.75)
        assert value == pytest.approx(3000.0 / 0.75)
