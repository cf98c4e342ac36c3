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


# ---------------------------------------------------------------------------------------
# one problem partitioned over two CPU ranks: heads, and sequence segments with the state
# exchange, each rank's arithmetic done by the oracle
# ---------------------------------------------------------------------------------------
def test_partition_helpers_cover_exactly():
    from chunkwise_causal_linear_gb300.shard import head_range, sequence_range
    for n in (0, 1, 7, 128):
        for world in (1, 2, 3, 8):
            parts = [head_range(n, world, r) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(parts, parts[1:]))
            sizes = [b - a for a, b in parts]
            assert max(sizes) - min(sizes) <= 1
    for L in (1, 63, 64, 1000, 8192):
        for world in (1, 2, 3, 5):
            segs = [sequence_range(L, world, r, 64) for r in range(world)]
            assert segs[0][0] == 0 and segs[-1][1] == L
            assert all(a[1] == b[0] for a, b in zip(segs, segs[1:]))
            assert all(a % 64 == 0 or a == b == L for a, b in segs)  # empty tail ranks


def _partition_rank(rank, world, port, q):
    import numpy as np

    import oracle
    import synth
    from chunkwise_causal_linear_gb300.shard import gather_totals, head_range, sequence_range
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = dict(synth.WORKLOADS["elu1-norm-d128-L8192"], B=1, H=3, L=700, dk=16, dv=24)
    inp = synth.make_inputs(w, seed=77)
    f64 = lambda x: synth.as_f64(x, w["dtype"])  # noqa: E731
    # heads: this rank's range, no communication
    h0, h1 = head_range(3, world, rank)
    heads_out = oracle.forward(f64(inp["q"][h0:h1]), f64(inp["k"][h0:h1]), f64(inp["v"][h0:h1]),
                               fm="elu1", normalize=True)
    # sequence: this rank's rows of every head; its own totals, gathered, then the prefix
    t0, t1 = sequence_range(w["L"], world, rank, 64)
    seg_out = []
    for h in range(3):
        fq = oracle.phi(f64(inp["q"][h, t0:t1]), "elu1")
        fk = oracle.phi(f64(inp["k"][h, t0:t1]), "elu1")
        vv = f64(inp["v"][h, t0:t1])
        _, T, zt = oracle.state_recurrence(fq, fk, vv, normalize=True, return_state=True)
        Ss, zs, rows = gather_totals(torch.from_numpy(T), torch.from_numpy(zt), t1 - t0)
        assert sum(rows) == w["L"]
        P = sum((Ss[r].numpy() for r in range(rank)), np.zeros_like(T))
        Pz = sum((zs[r].numpy() for r in range(rank)), np.zeros_like(zt))
        seg_out.append(oracle.state_recurrence(fq, fk, vv, normalize=True, S0=P, z0=Pz))
    q.put((rank, (h0, h1), heads_out, (t0, t1), np.stack(seg_out)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_partition_one_problem():
    """Two gloo ranks split one problem (B1 H3 L700, elu+1 with the normaliser) by heads and
    by sequence segments; the assembled outputs equal the oracle over the whole problem."""
    import numpy as np

    import oracle
    import synth
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_partition_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=120) for _ in range(2)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = dict(synth.WORKLOADS["elu1-norm-d128-L8192"], B=1, H=3, L=700, dk=16, dv=24)
    inp = synth.make_inputs(w, seed=77)
    f64 = lambda x: synth.as_f64(x, w["dtype"])  # noqa: E731
    ref = oracle.forward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), fm="elu1", normalize=True)
    heads = np.concatenate([g[2] for g in got], axis=0)
    assert [g[1] for g in got] == [(0, 2), (2, 3)]
    np.testing.assert_allclose(heads, ref, rtol=0, atol=1e-12 * np.abs(ref).max())
    seq = np.concatenate([g[4] for g in got], axis=1)
    assert [g[3] for g in got] == [(0, 384), (384, 700)]
    np.testing.assert_allclose(seq, ref, rtol=0, atol=1e-12 * np.abs(ref).max())
