"""The benchmark's multi-rank bookkeeping on CPU ranks (gloo, world size 2).

Heads are independent problems, so under torchrun every rank runs its own copy of the
workload (weak scaling) and no collective touches the data path; the only cross-rank step
is the max over ranks of the timed region.  This checks that step and the whole-job value
with two real processes.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t_ms = [12.5, 20.0][rank]            # rank 1 is the slow one
    worst = bench.max_over_ranks(dist, t_ms)
    value = bench.job_throughput(world, 1000, 5, worst)
    q.put((rank, worst, value))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, worst, value in got:
        assert worst == 20.0
        assert value == pytest.approx(2 * 1000 * 5 / 0.020)


def test_single_process_is_its_own_max():
    import bench
    assert bench.max_over_ranks(None, 3.25) == 3.25
    assert bench.job_throughput(1, 10, 2, 1000.0) == pytest.approx(20.0)
