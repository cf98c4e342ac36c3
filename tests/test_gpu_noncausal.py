"""Bidirectional (non-causal) linear attention, la_noncausal_fwd, against the oracle.

Every query sees every key ("Linear Attention / Performerの理論と実装", the non-causal
normalised form and the Performer's bidirectional FAVOR+; "attention と線形の間" section 1):
the oracle computes it state first; the pins tie that to plain matrix products.
"""
import numpy as np
import pytest

import synth
from parity_util import assert_close, oracle_heads, to_device, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunkwise_causal_linear_gb300 import build
    build.build()


def run_nc(w, inp):
    import torch

    import chunkwise_causal_linear_gb300 as la
    B, H, L, dk, dv = w["B"], w["H"], w["L"], w["dk"], w["dv"]
    q = to_device(inp["q"], w["dtype"], (B, H, L, dk))
    k = to_device(inp["k"], w["dtype"], (B, H, L, dk))
    v = to_device(inp["v"], w["dtype"], (B, H, L, dv))
    omega = None if inp["omega"] is None else torch.from_numpy(inp["omega"]).cuda()
    out = la.noncausal_fwd(q, k, v, feature_map=w["fm"], omega=omega, normalize=w["normalize"])
    torch.cuda.synchronize()
    st = la.la_last_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == la.LA_OK, la.la_status_string(st)
    return out.float().reshape(B * H, L, dv).double().cpu().numpy()


def oracle_nc(w, inp):
    import oracle
    q = synth.as_f64(inp["q"], w["dtype"])
    k = synth.as_f64(inp["k"], w["dtype"])
    v = synth.as_f64(inp["v"], w["dtype"])
    om = None if inp["omega"] is None else inp["omega"].astype(np.float64)
    return oracle.forward(q, k, v, fm=w["fm"], omega=om, normalize=w["normalize"], causal=False)


CASES = [
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=777)),            # tensor cores, ragged
    ("identity-d64-L2048", dict(B=1, H=2, L=2048)),             # tensor cores, split sequence
    ("identity-d64-L2048", dict(B=1, H=3, L=1000, normalize=True, fm="elu1", scale=1.0)),
    ("favor-m256-d64-L16384", dict(B=1, H=2, L=600)),           # Performer, tensor cores
    ("favor-m256-d64-L16384", dict(B=1, H=2, L=4096)),          # Performer, split sequence
    ("favor-m256-d64-L16384", dict(B=1, H=1, L=777, normalize=False)),
    ("favor-m256-d64-L16384", dict(B=1, H=2, L=100, dtype="f32")),  # Performer, generic path
    ("elu1-norm-d128-L8192", dict(B=2, H=1, L=100, dk=32, dv=48)),  # generic path
    # tensor cores: each branch of the main pass (Q-only tiles, z rows written once)
    ("identity-d64-L2048", dict(B=1, H=2, L=1500, normalize=True, dist="uniform01")),
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=1100, normalize=False)),
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=1000, dk=64, dv=128)),
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=4000)),            # split sequence, ragged
]


@pytest.mark.parametrize("base,over", CASES)
def test_noncausal_matches_oracle(base, over):
    w = workload(base, **over)
    inp = synth.make_inputs(w, seed=8)
    assert_close(run_nc(w, inp), oracle_nc(w, inp), f"non-causal {base} {over}")


def test_noncausal_integers_exact():
    w = workload("tiny-int-exact", B=2, H=1, L=50, dk=8, dv=12)
    inp = synth.make_inputs(w, seed=9)
    out, ref = run_nc(w, inp), oracle_nc(w, inp)
    assert np.array_equal(out, ref), np.abs(out - ref).max()


def test_noncausal_last_row_equals_causal_last_row():
    """The last query sees every key in both forms ("attention と線形の間" section 2)."""
    from parity_util import run_gpu
    w = workload("elu1-norm-d128-L8192", B=1, H=2, L=640)
    inp = synth.make_inputs(w, seed=10)
    nc = run_nc(w, inp)
    ca, _ = run_gpu(w, inp, 64, 0)
    assert_close(nc[:, -1:], ca[:, -1:], "last rows")


@pytest.mark.parametrize("name", ["elu1-norm-d128-L8192", "favor-m256-d64-L16384"])
def test_noncausal_full_size_all_outputs(name):
    """The benchmark's workloads (B8 H16 L8192 d128 elu+1 + normaliser; B2 H12 L16384 FAVOR+
    m=256): every head and row against the oracle's state-first form, and sampled rows of the
    first and last head against its definition (scores first)."""
    from parity_util import sample_rows
    w = workload(name)
    inp = synth.make_inputs(w, seed=12)
    out = run_nc(w, inp)
    assert_close(out, oracle_nc(w, inp), f"non-causal full size {name}, all outputs")
    heads = [0, w["B"] * w["H"] - 1]
    rows = sample_rows(w["L"], 64, 48, seed=12)
    import oracle
    f = lambda x: synth.as_f64(x[heads], w["dtype"])  # noqa: E731
    om = None if inp["omega"] is None else inp["omega"].astype(np.float64)
    ref = oracle.forward(f(inp["q"]), f(inp["k"]), f(inp["v"]), fm=w["fm"], omega=om,
                         normalize=w["normalize"], causal=False, method="scores_first", rows=rows)
    assert_close(out[heads][:, rows], ref, f"non-causal full size {name}, sampled rows")
