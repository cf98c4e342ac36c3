"""Carried state: la_chunked_state, la_state_combine, la_chunked_fwd_init.

A sequence cut into segments, each run from the prefix of the earlier segments' final
states ("attention と線形の間" section 2: the chunk scan at segment granularity), must give
the rows of one pass over the whole sequence; a prefill's final state must seed decoding.
Everything is checked against the oracle's pass over the whole sequence.
"""
import threading

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


def _tensors(w, inp):
    import torch
    B, H, L, dk, dv = w["B"], w["H"], w["L"], w["dk"], w["dv"]
    q = to_device(inp["q"], w["dtype"], (B, H, L, dk))
    k = to_device(inp["k"], w["dtype"], (B, H, L, dk))
    v = to_device(inp["v"], w["dtype"], (B, H, L, dv))
    om = None if inp["omega"] is None else torch.from_numpy(inp["omega"]).cuda()
    return q, k, v, om


def oracle_rows(w, inp, gamma):
    import oracle
    f = lambda x: synth.as_f64(x, w["dtype"])  # noqa: E731
    om = None if inp["omega"] is None else inp["omega"].astype(np.float64)
    return oracle.forward(f(inp["q"]), f(inp["k"]), f(inp["v"]), fm=w["fm"], omega=om,
                          normalize=w["normalize"], gamma=None if gamma == 1.0 else gamma)


def segmented(w, inp, cuts, gamma, C):
    """Rows of the whole sequence from per-segment passes started at the prefix state."""
    import torch

    import chunkwise_causal_linear_gb300 as la
    q, k, v, om = _tensors(w, inp)
    B, H, dv = w["B"], w["H"], w["dv"]
    D = om.shape[0] if om is not None else w["dk"]
    P = torch.zeros((B, H, D, dv), dtype=torch.float32, device="cuda")
    Pz = torch.zeros((B, H, D), dtype=torch.float32, device="cuda")
    outs = []
    s = torch.cuda.current_stream().cuda_stream
    bounds = [0] + list(cuts) + [w["L"]]
    for a, b in zip(bounds[:-1], bounds[1:]):
        qs, ks, vs = (x[:, :, a:b].contiguous() for x in (q, k, v))
        outs.append(la.chunked_fwd_init(qs, ks, vs, P, Pz, C=C, feature_map=w["fm"], omega=om,
                                        normalize=w["normalize"], gamma=gamma))
        T, Tz = la.chunked_state(ks, vs, feature_map=w["fm"], omega=om, gamma=gamma)
        # P <- gamma^len P + T: the prefix for the next segment
        rc = la.la_state_combine(P.data_ptr(), Pz.data_ptr(), T.data_ptr(), Tz.data_ptr(), B, H, D,
                                 dv, float(gamma ** (b - a)), s)
        assert rc == la.LA_OK
    torch.cuda.synchronize()
    st = la.la_last_device_status(s)
    assert st == la.LA_OK, la.la_status_string(st)
    return from_device(torch.cat(outs, dim=2)).reshape(B * H, w["L"], dv)


CASES = [
    # (base, overrides, cuts, gamma, C)
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=777), (300, 555), 1.0, 64),    # tensor cores
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=777), (300, 555), 0.95, 64),   # decay, tensor cores
    ("identity-d64-L2048", dict(B=1, H=2, L=600), (256,), 1.0, 16),          # C = 16
    ("identity-d64-L2048", dict(B=1, H=2, L=700, normalize=True, fm="elu1", scale=1.0), (129, 400), 1.0, 128),
    ("favor-m256-d64-L16384", dict(B=1, H=2, L=300), (100, 170), 1.0, 64),   # generic path
    ("identity-d64-L2048", dict(B=1, H=2, L=200, dtype="f32"), (50, 123), 0.9, 10),
]


@pytest.mark.parametrize("base,over,cuts,gamma,C", CASES)
def test_segments_compose_to_one_pass(base, over, cuts, gamma, C):
    w = workload(base, **over)
    inp = synth.make_inputs(w, seed=51)
    got = segmented(w, inp, cuts, gamma, C)
    assert_close(got, oracle_rows(w, inp, gamma), f"segments {base} {over} cuts={cuts} gamma={gamma}")


def test_final_state_matches_oracle():
    """la_chunked_state against the oracle's state after its recurrence (plain mask)."""
    import oracle

    import chunkwise_causal_linear_gb300 as la
    w = workload("elu1-norm-d128-L8192", B=1, H=2, L=333, dk=64, dv=64)
    inp = synth.make_inputs(w, seed=52)
    _, k, v, _ = _tensors(w, inp)
    S, z = la.chunked_state(k, v, feature_map="elu1")
    import torch
    torch.cuda.synchronize()
    for h in range(2):
        fk = oracle.phi(synth.as_f64(inp["k"][h], "bf16"), "elu1")
        fq = fk  # only the state is compared
        _, Sr, zr = oracle.state_recurrence(fq, fk, synth.as_f64(inp["v"][h], "bf16"),
                                            normalize=True, return_state=True)
        assert_close(from_device(S).reshape(2, 64, 64)[h], Sr, "state")
        assert_close(from_device(z).reshape(2, 64)[h], zr, "zstate")


@pytest.mark.parametrize("gamma", [1.0, 0.9])
def test_prefill_then_decode(gamma):
    """The state after a prefill of P rows seeds decoding rows P..L-1."""
    import torch

    import chunkwise_causal_linear_gb300 as la
    w = workload("elu1-norm-d128-L8192", B=2, H=2, L=320, dk=64, dv=64)
    inp = synth.make_inputs(w, seed=53)
    q, k, v, _ = _tensors(w, inp)
    Pn = 256
    S, z = la.chunked_state(k[:, :, :Pn].contiguous(), v[:, :, :Pn].contiguous(),
                            feature_map="elu1", gamma=gamma)
    rows = []
    for t in range(Pn, w["L"]):
        args = (q[:, :, t].contiguous(), k[:, :, t].contiguous(), v[:, :, t].contiguous())
        if gamma == 1.0:
            rows.append(la.decode_step(*args, S, z, t=t, feature_map="elu1", normalize=True))
        else:
            rows.append(la.decay_decode_step(*args, S, gamma, zstate=z, feature_map="elu1",
                                             normalize=True))
    got = from_device(torch.stack(rows, dim=2)).reshape(4, w["L"] - Pn, 64)
    ref = oracle_rows(w, inp, gamma)[:, Pn:]
    assert_close(got, ref, f"prefill + decode gamma={gamma}")


def test_host_thread_ranks_exchange_totals():
    """Two host threads, each with its own stream, own one half of the sequence: each
    computes its segment's total, the totals are exchanged through pinned host buffers, and
    each rank runs its half from the exclusive prefix (a two-rank sequence split on one GPU)."""
    import torch

    import chunkwise_causal_linear_gb300 as la
    gamma = 0.97
    w = workload("elu1-norm-d128-L8192", B=1, H=2, L=640)
    inp = synth.make_inputs(w, seed=54)
    q, k, v, _ = _tensors(w, inp)
    B, H, D, dv, half = 1, 2, 128, 128, 320
    host_T = [torch.empty((B, H, D, dv), dtype=torch.float32).pin_memory() for _ in range(2)]
    host_z = [torch.empty((B, H, D), dtype=torch.float32).pin_memory() for _ in range(2)]
    outs = [None, None]
    ready = [threading.Event(), threading.Event()]
    errors = []

    def rank(r):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                sl = slice(r * half, (r + 1) * half)
                qs, ks, vs = (x[:, :, sl].contiguous() for x in (q, k, v))
                T, Tz = la.chunked_state(ks, vs, feature_map="elu1", gamma=gamma,
                                         stream=stream.cuda_stream)
                host_T[r].copy_(T, non_blocking=True)
                host_z[r].copy_(Tz, non_blocking=True)
                stream.synchronize()
                ready[r].set()
                P = torch.zeros((B, H, D, dv), dtype=torch.float32, device="cuda")
                Pz = torch.zeros((B, H, D), dtype=torch.float32, device="cuda")
                if r == 1:  # exclusive prefix: rank 0's total
                    ready[0].wait(timeout=60)
                    P.copy_(host_T[0], non_blocking=True)
                    Pz.copy_(host_z[0], non_blocking=True)
                outs[r] = la.chunked_fwd_init(qs, ks, vs, P, Pz, feature_map="elu1",
                                              normalize=True, gamma=gamma,
                                              stream=stream.cuda_stream)
                stream.synchronize()
        except Exception as e:  # reported by the main thread
            errors.append(e)

    th = [threading.Thread(target=rank, args=(r,)) for r in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join(timeout=120)
    assert not errors, errors
    got = from_device(torch.cat(outs, dim=2)).reshape(2, w["L"], dv)
    assert_close(got, oracle_rows(w, inp, gamma), "two host-thread ranks")


def test_state_arguments():
    import torch

    import chunkwise_causal_linear_gb300 as la
    S = torch.zeros(1, 1, 8, 8, device="cuda")
    z = torch.zeros(1, 1, 8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert la.la_state_combine(S.data_ptr(), z.data_ptr(), S.data_ptr(), z.data_ptr(), 1, 1, 8, 8,
                               1.5, s) == la.LA_ERR_ARG
    assert la.la_state_combine(S.data_ptr(), None, S.data_ptr(), z.data_ptr(), 1, 1, 8, 8, 1.0,
                               s) == la.LA_ERR_NULL
    fav = la.make_feature_map("favor", 16, 0)
    k = torch.zeros(1, 1, 64, 8, device="cuda", dtype=torch.bfloat16)
    assert la.la_chunked_state(k.data_ptr(), k.data_ptr(), S.data_ptr(), None, 1, 1, 64, 8, 8, fav,
                               1.0, la.LA_BF16, s) == la.LA_ERR_NULL
