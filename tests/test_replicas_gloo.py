"""bench.py's multi-GPU path is replicas only (requests are independent; no
data-path collective): every rank runs the whole step on its own inputs, the
timings are reduced to their maximum over the ranks, and the job's throughput
counts the units of all ranks.  Checked here with two gloo ranks on the CPU,
through the functions bench.py itself uses."""
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


def _rank(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r saw (1 + r) ms for the timed steps and (5 - r) ms end to end
    ms, e2e = bench.max_over_ranks([1.0 + rank, 5.0 - rank], world, "cpu")
    out.put((rank, ms, e2e, bench.replica_throughput(128, world, 10, ms)))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for rank, ms, e2e, value in res:
        assert ms == 2.0 and e2e == 5.0, (rank, ms, e2e)
        # 128 units per step on each of 2 ranks, 10 steps in 2 ms
        assert value == pytest.approx(128 * 2 * 10 / 2e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0], 1, "cpu") == [3.0, 4.0]
    assert bench.replica_throughput(32, 1, 100, 50.0) == pytest.approx(32 * 100 / 0.05)
