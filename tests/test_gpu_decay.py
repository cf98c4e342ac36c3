"""Causal linear attention with the Retention decay (la_decay_fwd, la_decay_decode_step)
against the oracle.

The update S_t = gamma S_{t-1} + phi(k_t) v_t^T ("Linear Attention / Performerの理論と実装",
the section on the RNN without forgetting), z decaying alike under the normaliser; the
oracle runs the recurrence (or, for sampled rows of large problems, the weighted sum over
the past), and its pins tie both to closed forms and numpy.
"""
import numpy as np
import pytest

import synth
from parity_util import assert_close, from_device, to_device, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunkwise_causal_linear_gb300 import build
    build.build()


def _dev(w, inp):
    B, H, L, dk, dv = w["B"], w["H"], w["L"], w["dk"], w["dv"]
    return (to_device(inp["q"], w["dtype"], (B, H, L, dk)),
            to_device(inp["k"], w["dtype"], (B, H, L, dk)),
            to_device(inp["v"], w["dtype"], (B, H, L, dv)))


def run_decay(w, inp, gamma, path=0, C=64):
    import torch

    import chunkwise_causal_linear_gb300 as la
    q, k, v = _dev(w, inp)
    out = la.decay_fwd(q, k, v, gamma, C=C, feature_map=w["fm"], normalize=w["normalize"],
                       path=path)
    torch.cuda.synchronize()
    st = la.la_last_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == la.LA_OK, la.la_status_string(st)
    return from_device(out).reshape(w["B"] * w["H"], w["L"], w["dv"])


def oracle_decay(w, inp, gamma, heads=None, rows=None):
    import oracle
    sel = slice(None) if heads is None else heads
    q = synth.as_f64(inp["q"][sel], w["dtype"])
    k = synth.as_f64(inp["k"][sel], w["dtype"])
    v = synth.as_f64(inp["v"][sel], w["dtype"])
    method = "recurrence" if rows is None else "scores_first"
    return oracle.forward(q, k, v, fm=w["fm"], normalize=w["normalize"], gamma=gamma,
                          method=method, rows=rows)


def plan_path(w, gamma, path=0, C=64):
    import chunkwise_causal_linear_gb300 as la
    fm = la.make_feature_map(w["fm"])
    dt = la.LA_BF16 if w["dtype"] == "bf16" else la.LA_F32
    rc, info = la.la_decay_plan(w["B"], w["H"], w["L"], w["dk"], w["dv"], C, fm,
                                int(w["normalize"]), gamma, dt, path, 0)
    return rc, info


# (base workload, overrides, gamma, path): 0 auto, 1 generic, 2 tensor cores
CASES = [
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=777), 0.98, 2),           # ragged tail
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=777, normalize=False, scale=0.3), 0.9, 2),
    ("identity-d64-L2048", dict(B=1, H=3, L=1000), 0.95, 2),
    ("identity-d64-L2048", dict(B=1, H=2, L=640, dv=128), 0.7, 2),
    ("identity-d64-L2048", dict(B=1, H=2, L=640, normalize=True, fm="elu1", scale=1.0), 0.5, 2),
    # gamma = 0.75: the fp32 state is rescaled every second chunk
    ("identity-d64-L2048", dict(B=1, H=2, L=640, normalize=True, fm="elu1", scale=1.0), 0.75, 2),
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=700, normalize=False, scale=0.3), 0.75, 2),
    ("identity-d64-L2048", dict(B=1, H=2, L=2048), 0.99, 2),             # split sequence
    ("elu1-norm-d128-L8192", dict(B=1, H=1, L=4096), 0.999, 2),          # split sequence
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=300), 0.3, 0),             # gamma < 0.5: generic
    ("elu1-norm-d128-L8192", dict(B=2, H=1, L=200, dk=32, dv=48), 0.9, 0),  # generic dims
    ("identity-d64-L2048", dict(B=1, H=2, L=333, dtype="f32"), 0.8, 1),  # generic fp32
]


@pytest.mark.parametrize("base,over,gamma,path", CASES)
def test_decay_matches_oracle(base, over, gamma, path):
    w = workload(base, **over)
    inp = synth.make_inputs(w, seed=21)
    rc, info = plan_path(w, gamma, path)
    assert rc == 0
    if path == 0 and gamma < 0.5:
        assert info["path"] == 1  # the tensor cores need gamma^64 >= 2^-64
    out = run_decay(w, inp, gamma, path)
    assert_close(out, oracle_decay(w, inp, gamma), f"decay {base} {over} gamma={gamma}")


@pytest.mark.parametrize("C", [1, 16, 64, 100])
def test_decay_generic_fp32_tight(C):
    """fp32 storage on the generic path: errors at fp32 rounding level for any chunk size
    (the decay factors come from exp2 of log2(gamma) times an integer)."""
    w = workload("tiny-int-exact", B=2, H=1, L=203, dk=16, dv=24, dist="normal", scale=0.5)
    inp = synth.make_inputs(w, seed=22)
    out = run_decay(w, inp, 0.93, path=1, C=C)
    ref = oracle_decay(w, inp, 0.93)
    err = np.abs(out - ref).max() / np.abs(ref).max()
    assert err < 2e-6, err


@pytest.mark.parametrize("path", [1, 2])
def test_decay_gamma_one_equals_plain(path):
    """gamma = 1 multiplies by exact ones: the result equals la_chunked_fwd's bit for bit
    on the same path."""
    from parity_util import run_gpu
    base = "elu1-norm-d128-L8192" if path == 2 else "tiny-int-exact"
    w = workload(base, B=1, H=2, L=640)
    inp = synth.make_inputs(w, seed=23)
    a = run_decay(w, inp, 1.0, path)
    b, _ = run_gpu(w, inp, 64, path)
    assert np.array_equal(a, b)


def test_decay_full_size_all_outputs():
    """The decayed workload at full size (B=8, H=16, L=8192, d=128, elu+1, normaliser,
    gamma = 0.98) on the tensor cores, as the benchmark runs it: every head and row against
    the oracle's recurrence, and sampled rows of three heads against its weighted sum over
    the past."""
    w = workload("decay-elu1-norm-d128-L8192")
    gamma = w["gamma"]
    rc, info = plan_path(w, gamma)
    assert rc == 0 and info["path"] == 2
    inp = synth.make_inputs(w, seed=24)
    out = run_decay(w, inp, gamma)
    assert_close(out, oracle_decay(w, inp, gamma), "full-size decay, all outputs")
    heads = [0, 77, 127]
    rows = [0, 1, 63, 64, 65, 4095, 4096, 8190, 8191]
    ref = oracle_decay(w, {k: (v[heads] if isinstance(v, np.ndarray) else v)
                           for k, v in inp.items()}, gamma, rows=rows)
    assert_close(out[heads][:, rows], ref, "full-size decay sampled rows")


def test_decay_rejects_bad_gamma():
    import torch

    import chunkwise_causal_linear_gb300 as la
    w = workload("identity-d64-L2048", B=1, H=1, L=128)
    inp = synth.make_inputs(w, seed=25)
    q, k, v = _dev(w, inp)
    out = torch.empty_like(v)
    fm = la.make_feature_map("identity")
    s = torch.cuda.current_stream().cuda_stream
    for g in (0.0, -0.5, 1.5, float("nan")):
        rc = la.la_decay_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), 1, 1, 128,
                             64, 64, 64, fm, 0, g, la.LA_BF16, None, 0, s, 0)
        assert rc == la.LA_ERR_ARG, g
    # gamma below 0.5 is not on the tensor cores
    rc = la.la_decay_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), 1, 1, 128, 64,
                         64, 64, fm, 0, 0.4, la.LA_BF16, None, 0, s, la.LA_PATH_TC)
    assert rc == la.LA_ERR_UNSUPPORTED


@pytest.mark.parametrize("fm,normalize,dv", [("identity", False, 64), ("elu1", True, 128),
                                              ("elu1", True, 20)])
def test_decay_decode_steps_reproduce_forward(fm, normalize, dv):
    """Stepping la_decay_decode_step over t = 0..L-1 from zero state gives the forward
    rows (and the oracle's)."""
    import torch

    import chunkwise_causal_linear_gb300 as la
    gamma = 0.9
    w = workload("elu1-norm-d128-L8192", B=2, H=2, L=96, dk=64, dv=dv, fm=fm,
                 normalize=normalize, scale=0.5)
    inp = synth.make_inputs(w, seed=26)
    q, k, v = _dev(w, inp)
    S, z = la.decode_state(2, 2, 64, dv, feature_map=fm, normalize=normalize)
    rows = []
    for t in range(w["L"]):
        o = la.decay_decode_step(q[:, :, t].contiguous(), k[:, :, t].contiguous(),
                                 v[:, :, t].contiguous(), S, gamma, zstate=z, feature_map=fm,
                                 normalize=normalize)
        rows.append(o)
    dec = torch.stack(rows, dim=2)
    torch.cuda.synchronize()
    got = from_device(dec).reshape(4, w["L"], dv)
    assert_close(got, oracle_decay(w, inp, gamma), "decay decode vs oracle")
    fwd = run_decay(w, inp, gamma, path=1)
    assert_close(got, fwd, "decay decode vs forward")
