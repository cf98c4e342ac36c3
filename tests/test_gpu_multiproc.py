"""One problem split over two processes that exchange data through torch.distributed (gloo),
both on the one GPU: the multi-process form of the library's two partitions.

* Heads: each rank runs la_chunked_fwd on its own contiguous range of heads.
* Sequence: each rank owns a contiguous range of rows of the same heads, computes its
  segment's total with la_chunked_state, the ranks all-gather the fp32 totals, and each
  rank starts la_chunked_fwd_init from the exclusive prefix of the earlier totals
  (la_state_combine), as ``chunkwise_causal_linear_gb300.shard.sequence_parallel_fwd`` does
  ("attention と線形の間" section 2: the carried state at segment granularity).

The kernels of the two processes never wait on one another: the only exchange is the
host-side all-gather between their launches.  The assembled output is compared with the
oracle over the whole problem.
"""
import os
import socket

import numpy as np
import pytest

import synth
from parity_util import assert_close, oracle_heads, workload

pytestmark = pytest.mark.gpu

# (workload, overrides, gamma): plain mask with the normaliser, and the Retention decay
CASES = [
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=1500), 1.0),
    ("identity-d64-L2048", dict(B=2, H=2, L=1000), 0.98),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunkwise_causal_linear_gb300 import build
    build.build()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, outdir):
    import torch
    import torch.distributed as dist

    import chunkwise_causal_linear_gb300 as la
    from chunkwise_causal_linear_gb300.shard import head_range, sequence_parallel_fwd, sequence_range
    from parity_util import to_device
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    for i, (base, over, gamma) in enumerate(CASES):
        w = workload(base, **over)
        B, H, L, dk, dv = w["B"], w["H"], w["L"], w["dk"], w["dv"]
        inp = synth.make_inputs(w, seed=51 + i)
        q = to_device(inp["q"], w["dtype"], (B, H, L, dk))
        k = to_device(inp["k"], w["dtype"], (B, H, L, dk))
        v = to_device(inp["v"], w["dtype"], (B, H, L, dv))
        # sequence segments of every head
        t0, t1 = sequence_range(L, world, rank, 64)
        seg = lambda x: x[:, :, t0:t1].contiguous()  # noqa: E731
        o = sequence_parallel_fwd(seg(q), seg(k), seg(v), C=64, feature_map=w["fm"],
                                  normalize=w["normalize"], gamma=gamma)
        torch.cuda.synchronize()
        st = la.la_last_device_status(torch.cuda.current_stream().cuda_stream)
        assert st == la.LA_OK, la.la_status_string(st)
        np.save(os.path.join(outdir, f"seq{i}_r{rank}.npy"),
                o.to(torch.float64).cpu().numpy().reshape(B * H, t1 - t0, dv))
        # heads: this rank's range of the flattened B*H heads (gamma = 1 cases only)
        if gamma == 1.0:
            h0, h1 = head_range(B * H, world, rank)
            flat = lambda x: x.reshape(B * H, L, -1)[h0:h1].unsqueeze(0).contiguous()  # noqa: E731
            oh = la.chunked_fwd(flat(q), flat(k), flat(v), C=64, feature_map=w["fm"],
                                normalize=w["normalize"])
            torch.cuda.synchronize()
            np.save(os.path.join(outdir, f"heads{i}_r{rank}.npy"),
                    oh.to(torch.float64).cpu().numpy().reshape(h1 - h0, L, dv))
    dist.barrier()
    dist.destroy_process_group()


def test_two_processes_split_one_problem(tmp_path):
    import torch.multiprocessing as mp

    from chunkwise_causal_linear_gb300.shard import sequence_range
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    for i, (base, over, gamma) in enumerate(CASES):
        w = workload(base, **over)
        inp = synth.make_inputs(w, seed=51 + i)
        n = w["B"] * w["H"]
        if gamma == 1.0:
            ref = oracle_heads(w, inp, list(range(n)), method="recurrence")
        else:
            import oracle
            f = lambda x: synth.as_f64(x, w["dtype"])  # noqa: E731
            ref = oracle.forward(f(inp["q"]), f(inp["k"]), f(inp["v"]), fm=w["fm"],
                                 normalize=w["normalize"], gamma=gamma)
        parts = [np.load(tmp_path / f"seq{i}_r{r}.npy") for r in range(2)]
        assert [p.shape[1] for p in parts] == [b - a for a, b in
                                               (sequence_range(w["L"], 2, r, 64) for r in range(2))]
        assert_close(np.concatenate(parts, axis=1), ref, f"sequence split {base} {over}")
        if gamma == 1.0:
            heads = np.concatenate([np.load(tmp_path / f"heads{i}_r{r}.npy") for r in range(2)])
            assert_close(heads, ref, f"heads split {base} {over}")
