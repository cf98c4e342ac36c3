"""Backward pass (la_chunked_bwd) against the oracle's gradients.

The oracle applies the chain rule to the plain causal definition (pinned by finite
differences of its forward recurrence); the library composes causal and anti-causal
linear-attention passes, on the generic fp32 path or on the tensor cores.
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


def run_bwd(w, inp, dout_bits, C, gamma=1.0, path=0):
    import torch

    import chunkwise_causal_linear_gb300 as la
    B, H, L, dk, dv = w["B"], w["H"], w["L"], w["dk"], w["dv"]
    q = to_device(inp["q"], w["dtype"], (B, H, L, dk))
    k = to_device(inp["k"], w["dtype"], (B, H, L, dk))
    v = to_device(inp["v"], w["dtype"], (B, H, L, dv))
    do = to_device(dout_bits, w["dtype"], (B, H, L, dv))
    omega = None if inp["omega"] is None else torch.from_numpy(inp["omega"]).cuda()
    dq, dk_, dv_ = la.chunked_bwd(q, k, v, do, C=C, feature_map=w["fm"], omega=omega,
                                  normalize=w["normalize"], gamma=gamma, path=path)
    torch.cuda.synchronize()
    st = la.la_last_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == la.LA_OK, la.la_status_string(st)
    n = B * H
    return (from_device(dq).reshape(n, L, dk), from_device(dk_).reshape(n, L, dk),
            from_device(dv_).reshape(n, L, dv))


def oracle_bwd(w, inp, dout_bits, gamma=1.0):
    import oracle
    f = lambda x: synth.as_f64(x, w["dtype"])  # noqa: E731
    om = None if inp["omega"] is None else inp["omega"].astype(np.float64)
    return oracle.backward(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(dout_bits), fm=w["fm"],
                           omega=om, normalize=w["normalize"],
                           gamma=None if gamma == 1.0 else gamma)


def dout_for(w, seed):
    """The upstream gradient: seeded N(0,1) values in the storage dtype, [B*H, L, dv]."""
    return synth.tensor_values(seed, synth.T_DOUT, w["B"], w["H"], w["L"], w["dv"], "normal", 1.0,
                               w["dtype"])


CASES = [
    # (base workload, overrides, C, gamma)
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=333, dk=64, dv=64), 64, 1.0),
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=300, dk=32, dv=48, normalize=False), 16, 1.0),
    ("identity-d64-L2048", dict(B=2, H=1, L=257), 64, 1.0),
    ("identity-d64-L2048", dict(B=1, H=2, L=200), 100, 0.9),
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=190, dk=64, dv=64), 32, 0.95),
    ("favor-m256-d64-L16384", dict(B=1, H=2, L=150), 64, 1.0),
    ("favor-m256-d64-L16384", dict(B=1, H=1, L=130, normalize=False), 64, 1.0),
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=2048), 64, 1.0),  # d128, 32 tiles per head
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=700, normalize=False), 64, 1.0),
    ("identity-d64-L2048", dict(B=1, H=3, L=1000, normalize=True, fm="elu1", scale=1.0), 64, 1.0),
    # the decay without the normaliser on the tensor-core route: split sequence, d128, d64
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=2048, normalize=False), 64, 0.98),
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=700, normalize=False), 64, 0.9),
    ("identity-d64-L2048", dict(B=2, H=2, L=777), 64, 0.75),
    # FAVOR+ on the tensor-core route: split sequence, m = 128 and 256, with and without the
    # normaliser
    ("favor-m256-d64-L16384", dict(B=1, H=2, L=1500), 64, 1.0),
    ("favor-m256-d64-L16384", dict(B=2, H=1, L=700, m=128, normalize=False), 64, 1.0),
    ("favor-m256-d64-L16384", dict(B=1, H=2, L=400, m=512), 64, 1.0),
]


def bwd_path(w, gamma):
    """1 (generic) or 2 (tensor cores): the path la_chunked_bwd takes on AUTO."""
    if w["dtype"] != "bf16" or w["L"] < 128:
        return 1
    if w["fm"] == "favor":
        return 2 if (gamma == 1.0 and w["dk"] == w["dv"] == 64 and w["m"] in (128, 256, 512)) else 1
    return 2 if (w["fm"] in ("identity", "elu1")
                 and (gamma == 1.0 or (gamma >= 0.5 and not w["normalize"]))
                 and w["dk"] == w["dv"] and w["dk"] in (64, 128)) else 1


@pytest.mark.parametrize("base,over,C,gamma", CASES)
def test_backward_matches_oracle(base, over, C, gamma):
    w = workload(base, **over)
    inp = synth.make_inputs(w, seed=41)
    do = dout_for(w, 41)
    ref = oracle_bwd(w, inp, do, gamma)
    paths = [1] + ([2] if bwd_path(w, gamma) == 2 else [])
    for path in paths:
        got = run_bwd(w, inp, do, C, gamma, path)
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert_close(g, r, f"{name} {base} {over} C={C} gamma={gamma} path={path}")


FULL_CASES = [
    # (benchmark workload, heads compared row by row; None: every head)
    ("elu1-norm-d128-L8192", (0, 63, 127)),
    ("identity-d64-L2048", None),
]


@pytest.mark.parametrize("base,heads", FULL_CASES)
def test_backward_full_size(base, heads):
    """The benchmark's backward workloads at full size, on the path AUTO takes (the tensor
    cores), against the oracle's gradients: every row and every output of the listed heads.
    The oracle's plain chain rule costs O(L^2 d) per head, about 20 s at L = 8192 and
    d = 128, so the default workload compares its first, a middle and its last head; the
    short-sequence workload compares all of them."""
    w = workload(base)
    inp = synth.make_inputs(w, seed=43)
    do = dout_for(w, 43)
    got = run_bwd(w, inp, do, 64, 1.0, 0)
    n = w["B"] * w["H"]
    hs = list(range(n)) if heads is None else list(heads)
    ref = oracle_bwd(w, synth.make_inputs(w, seed=43, heads=hs), do[hs])
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert_close(g[hs], r, f"{name} {base} full size, heads {hs}")


def test_backward_tensor_core_route_is_taken():
    """LA_PATH_TC succeeds where the route applies and is refused where it does not."""
    import torch

    import chunkwise_causal_linear_gb300 as la
    w = workload("elu1-norm-d128-L8192", B=1, H=2, L=256)
    inp = synth.make_inputs(w, seed=43)
    do = dout_for(w, 43)
    run_bwd(w, inp, do, 64, 1.0, path=2)
    wn = dict(w, normalize=False)
    run_bwd(wn, inp, do, 64, 0.9, path=2)      # decay with gamma >= 0.5, no normaliser: tensor cores
    with pytest.raises(la.LAError):
        run_bwd(w, inp, do, 64, 0.9, path=2)   # decay with the normaliser: generic path only
    with pytest.raises(la.LAError):
        run_bwd(wn, inp, do, 64, 0.4, path=2)  # gamma^64 below 2^-64: generic path only
    wf = workload("elu1-norm-d128-L8192", B=1, H=1, L=256, dtype="f32")
    inpf = synth.make_inputs(wf, seed=43)
    with pytest.raises(la.LAError):
        run_bwd(wf, inpf, dout_for(wf, 43), 64, 1.0, path=2)  # fp32 storage
    torch.cuda.synchronize()


@pytest.mark.parametrize("normalize", [False, True])
def test_backward_fp32_tight(normalize):
    """fp32 storage: gradients at fp32 rounding level, and independent of the chunk size."""
    w = workload("tiny-int-exact", B=1, H=2, L=150, dk=12, dv=10, dist="normal", scale=0.5,
                 fm="elu1", normalize=normalize)
    inp = synth.make_inputs(w, seed=42)
    do = dout_for(w, 42)
    ref = oracle_bwd(w, inp, do)
    runs = [run_bwd(w, inp, do, C) for C in (1, 16, 150)]
    for got in runs:
        for g, r in zip(got, ref):
            err = np.abs(g - r).max() / np.abs(r).max()
            assert err < 2e-5, err


def test_backward_rejects_bad_arguments():
    import torch

    import chunkwise_causal_linear_gb300 as la
    fm = la.make_feature_map("elu1")
    t = torch.zeros(1, 1, 64, 16, device="cuda", dtype=torch.bfloat16)
    p = t.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    args = (1, 1, 64, 16, 16, 64, fm)
    assert la.la_chunked_bwd(p, p, p, None, p, p, p, *args, 1, 1.0, la.LA_BF16, ws.data_ptr(),
                             ws.numel(), s) == la.LA_ERR_NULL
    assert la.la_chunked_bwd(p, p, p, p, p, p, p, *args, 0, 1.5, la.LA_BF16, ws.data_ptr(),
                             ws.numel(), s) == la.LA_ERR_ARG
    assert la.la_chunked_bwd(p, p, p, p, p, p, p, *args, 0, 1.0, la.LA_BF16, ws.data_ptr(), 16,
                             s) == la.LA_ERR_WORKSPACE


# ---------------------------------------------------------------------------------------
# log-linear mask ("論文紹介：Log Linear Attention", slide 17): la_chunked_bwd_ll
# ---------------------------------------------------------------------------------------
LL_CASES = [
    # (base workload, overrides): ragged lengths, several levels of chunk blocks, every map
    ("loglinear-d64-L65536", dict(B=1, H=2, L=1000)),
    ("loglinear-d64-L65536", dict(B=2, H=1, L=333, dk=32, dv=48)),
    ("loglinear-d64-L65536", dict(B=1, H=1, L=4096)),                       # 64 chunks, 6 block levels
    ("loglinear-d64-L65536", dict(B=1, H=2, L=700, fm="elu1", normalize=True, scale=1.0)),
    ("loglinear-d64-L65536", dict(B=1, H=2, L=200, fm="favor", m=256, normalize=True, scale=1.0)),
    ("loglinear-d64-L65536", dict(B=1, H=1, L=50)),                          # one chunk
    ("loglinear-d64-L65536", dict(B=1, H=2, L=300, dtype="f32")),
]


def run_bwd_ll(w, inp, dout_bits):
    import torch

    import chunkwise_causal_linear_gb300 as la
    B, H, L, dk, dv = w["B"], w["H"], w["L"], w["dk"], w["dv"]
    q = to_device(inp["q"], w["dtype"], (B, H, L, dk))
    k = to_device(inp["k"], w["dtype"], (B, H, L, dk))
    v = to_device(inp["v"], w["dtype"], (B, H, L, dv))
    do = to_device(dout_bits, w["dtype"], (B, H, L, dv))
    lam = torch.from_numpy(inp["lam"]).reshape(B, H, L, -1).cuda()
    omega = None if inp["omega"] is None else torch.from_numpy(inp["omega"]).cuda()
    dq, dk_, dv_ = la.chunked_bwd_ll(q, k, v, do, lam, C=64, feature_map=w["fm"], omega=omega,
                                     normalize=w["normalize"])
    torch.cuda.synchronize()
    st = la.la_last_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == la.LA_OK, la.la_status_string(st)
    n = B * H
    return (from_device(dq).reshape(n, L, dk), from_device(dk_).reshape(n, L, dk),
            from_device(dv_).reshape(n, L, dv))


@pytest.mark.parametrize("base,over", LL_CASES)
def test_loglinear_backward_matches_oracle(base, over):
    import oracle
    w = workload(base, **over)
    inp = synth.make_inputs(w, seed=61)
    do = dout_for(w, 61)
    f = lambda x: synth.as_f64(x, w["dtype"])  # noqa: E731
    om = None if inp["omega"] is None else inp["omega"].astype(np.float64)
    ref = oracle.backward(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(do), fm=w["fm"], omega=om,
                          normalize=w["normalize"], lam=inp["lam"].astype(np.float64))
    got = run_bwd_ll(w, inp, do)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        if w["dtype"] == "f32":
            # fp32 storage: errors at fp32 rounding level
            assert np.abs(g - r).max() <= 1e-4 * np.abs(r).max(), (name, np.abs(g - r).max())
        else:
            assert_close(g, r, f"{name} log-linear {over}")


def test_loglinear_backward_all_ones_equals_plain_backward():
    """lambda == 1 is the plain mask: la_chunked_bwd_ll equals la_chunked_bwd (generic path)
    to fp32 rounding."""
    import torch
    w = workload("loglinear-d64-L65536", B=1, H=2, L=900, dtype="f32")
    inp = synth.make_inputs(w, seed=62)
    inp["lam"] = np.ones_like(inp["lam"])
    do = dout_for(w, 62)
    a = run_bwd_ll(w, inp, do)
    b = run_bwd(dict(w, loglinear=False), dict(inp, lam=None), do, 64, 1.0, 1)
    for x, y in zip(a, b):
        assert np.abs(x - y).max() <= 1e-5 * np.abs(y).max()
    torch.cuda.synchronize()


def test_loglinear_backward_rejects_bad_arguments():
    import torch

    import chunkwise_causal_linear_gb300 as la
    fm = la.make_feature_map("identity")
    x = torch.zeros(1, 1, 256, 64, dtype=torch.bfloat16, device="cuda")
    lam = torch.ones(1, 1, 256, 9, device="cuda")
    p = x.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    need = la.la_chunked_bwd_ll_workspace_bytes(1, 1, 256, 64, 64, 64, fm, 0, 9, la.LA_BF16)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    # too few levels for 256 rows (1 + 8 = 9 needed)
    assert la.la_chunked_bwd_ll_workspace_bytes(1, 1, 256, 64, 64, 64, fm, 0, 8, la.LA_BF16) == 0
    rc = la.la_chunked_bwd_ll(p, p, p, p, p, p, p, 1, 1, 256, 64, 64, 64, fm, 0, lam.data_ptr(), 8,
                              la.LA_BF16, ws.data_ptr(), need, s)
    assert rc != la.LA_OK
    rc = la.la_chunked_bwd_ll(p, p, p, p, p, p, p, 1, 1, 256, 64, 64, 64, fm, 0, None, 9,
                              la.LA_BF16, ws.data_ptr(), need, s)
    assert rc == la.LA_ERR_NULL
    rc = la.la_chunked_bwd_ll(p, p, p, p, p, p, p, 1, 1, 256, 64, 64, 64, fm, 0, lam.data_ptr(), 9,
                              la.LA_BF16, ws.data_ptr(), need - 1, s)
    assert rc == la.LA_ERR_WORKSPACE
    rc = la.la_chunked_bwd_ll(p, p, p, p, p, p, p, 1, 1, 256, 64, 64, 64, fm, 0, lam.data_ptr(), 9,
                              la.LA_BF16, ws.data_ptr(), need, s, la.LA_PATH_TC)
    assert rc == la.LA_ERR_UNSUPPORTED
