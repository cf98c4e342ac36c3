"""GPU parity: the library (through its C ABI) against the CPU oracle, element by element.

Small cases and the full-size workloads compare every output with the oracle's
recurrence; the full-size workloads also compare sampled rows of two heads (first and
last 2C rows plus random rows) with the oracle's scores-first definition.  The integer case must be bit-exact; bf16
cases must satisfy max|err| <= 2e-2 max|ref| and ||err||/||ref|| <= 5e-3.
"""
import numpy as np
import pytest

import synth
from parity_util import (assert_close, from_device, oracle_heads, run_gpu, sample_rows, to_device,
                         workload)

pytestmark = pytest.mark.gpu

SIMT, TC, AUTO = 1, 2, 0


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunkwise_causal_linear_gb300 import build
    build.build()


def tc_supported(w, C):
    import chunkwise_causal_linear_gb300 as la
    fm = la.make_feature_map(w["fm"], w["m"], 1 if w["fm"] == "favor" else 0)
    nl = synth.num_levels(w["L"]) if w.get("loglinear") else 0
    rc, _ = la.la_chunked_plan(w["B"], w["H"], w["L"], w["dk"], w["dv"], C, fm,
                               int(w["normalize"]), int(bool(w.get("loglinear"))), nl,
                               la.LA_BF16 if w["dtype"] == "bf16" else la.LA_F32, TC, 0)
    return rc == la.LA_OK


def paths_for(w, C):
    return [SIMT] + ([TC] if tc_supported(w, C) else [])


# ---------------------------------------------------------------------------
# exactness case: integers in {-3..3}, fp32, identity, no normaliser
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("C", [1, 4, 16, 64, 0, -5, 3, 7, 100])
@pytest.mark.parametrize("path", [SIMT, AUTO])
def test_tiny_integer_case_bit_exact(C, path):
    w = workload("tiny-int-exact")
    inp = synth.make_inputs(w, seed=1)
    out, _ = run_gpu(w, inp, C, path)
    ref = oracle_heads(w, inp, [0], method="scores_first")
    assert np.array_equal(out, ref), np.abs(out - ref).max()


@pytest.mark.parametrize("L,C", [(50, 16), (50, 7), (1, 1), (1, 64), (129, 64), (64, 65)])
def test_integer_ragged_bit_exact(L, C):
    w = workload("tiny-int-exact", B=2, H=3, L=L, dk=8, dv=40)
    inp = synth.make_inputs(w, seed=2)
    out, _ = run_gpu(w, inp, C, SIMT)
    ref = oracle_heads(w, inp, list(range(6)), method="scores_first")
    assert np.array_equal(out, ref)


# ---------------------------------------------------------------------------
# reduced-size versions of each workload: full outputs against the oracle recurrence
# ---------------------------------------------------------------------------
SMALL = [
    ("identity-d64-L2048", dict(B=1, H=3, L=333), 64),
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=777), 16),
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=777), 32),
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=777), 64),
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=777), 128),
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=777), 256),
    ("favor-m256-d64-L16384", dict(B=1, H=2, L=600), 64),
    ("favor-m256-d64-L16384", dict(B=1, H=1, L=777, normalize=False), 64),
    # few heads: the tensor-core path splits each sequence into segments
    ("favor-m256-d64-L16384", dict(B=1, H=2, L=4096), 64),
    ("loglinear-d64-L65536", dict(B=1, H=2, L=1000), 64),
    # few heads: the tensor-core path splits the sequence; ragged last chunk
    ("loglinear-d64-L65536", dict(B=1, H=3, L=4096), 64),
    ("loglinear-d64-L65536", dict(B=2, H=2, L=2000), 64),
    ("loglinear-d64-L65536", dict(B=1, H=1, L=300), 16),
    ("loglinear-d64-L65536", dict(B=1, H=1, L=200), 1),
    ("elu1-norm-d128-L8192", dict(B=1, H=1, L=1, ), 64),
    ("elu1-norm-d128-L8192", dict(B=1, H=1, L=100, dk=32, dv=48), 64),
    ("identity-d64-L2048", dict(B=1, H=1, L=200, dk=16, dv=16), 64),
]


@pytest.mark.parametrize("base,over,C", SMALL)
def test_small_workloads_match_oracle(base, over, C):
    w = workload(base, **over)
    inp = synth.make_inputs(w, seed=3)
    n = w["B"] * w["H"]
    ref = oracle_heads(w, inp, list(range(n)), method="recurrence")
    for path in paths_for(w, C):
        out, _ = run_gpu(w, inp, C, path)
        assert_close(out, ref, f"{base} {over} C={C} path={path}")


@pytest.mark.parametrize("path", [SIMT, TC])
def test_loglinear_all_ones_equals_plain(path):
    """Slide 17 of the log-linear deck: lambda == 1 gives linear attention."""
    w = workload("loglinear-d64-L65536", B=1, H=2, L=500)
    inp = synth.make_inputs(w, seed=4)
    inp["lam"] = np.ones_like(inp["lam"])
    out_ll, _ = run_gpu(w, inp, 64, path)
    wp = dict(w, loglinear=False)
    inp_p = dict(inp, lam=None)
    out_p, _ = run_gpu(wp, inp_p, 64, SIMT)
    assert_close(out_ll, out_p, "lambda=1 vs plain")
    ref = oracle_heads(wp, inp_p, [0, 1])
    assert_close(out_ll, ref, "lambda=1 vs oracle")


# ---------------------------------------------------------------------------
# full-size workloads, in the configuration the benchmark times (automatic path)
# ---------------------------------------------------------------------------
FULL = [("identity-d64-L2048", 64), ("favor-m256-d64-L16384", 64),
        ("loglinear-d64-L65536", 64)] + [("elu1-norm-d128-L8192", C) for C in
                                         (16, 32, 64, 128, 256)]

_cache = {}


def full_reference(name):
    """Inputs and the oracle's whole output (state recurrence, all heads, threaded over
    heads) for a full-size workload.  The output does not depend on C, so the C sweep
    shares one oracle run."""
    if name not in _cache:
        _cache.clear()
        w = workload(name)
        inp = synth.make_inputs(w, seed=11)
        ref = oracle_heads(w, inp, list(range(w["B"] * w["H"])), method="recurrence")
        _cache[name] = (w, inp, ref)
    return _cache[name]


@pytest.mark.parametrize("name,C", FULL)
def test_full_size_all_outputs(name, C):
    """Every head and every row of the full-size workload, in the configuration the
    benchmark times, against the oracle's recurrence; sampled rows of two heads also
    against the scores-first definition (an independent order)."""
    w, inp, ref = full_reference(name)
    out, _ = run_gpu(w, inp, C, AUTO)
    assert_close(out, ref, f"{name} C={C} all outputs")
    n = w["B"] * w["H"]
    heads = [0, n - 1]
    rows = sample_rows(w["L"], C, 48, seed=C)
    ref_sf = oracle_heads(w, inp, heads, method="scores_first", rows=rows)
    assert_close(out[heads][:, rows], ref_sf, f"{name} C={C} sampled rows")


HOST_CASES = [
    # (workload, overrides): pipelined over head groups (>= 64 MB moved), or one sequence
    ("elu1-norm-d128-L8192", dict(L=2048)),             # 128 heads, 268 MB: 8 groups of 16
    ("elu1-norm-d128-L8192", dict(B=3, H=27, L=1000)),  # 81 heads: 7 groups of 11 and one of 4
    ("identity-d64-L2048", dict()),                     # 33 MB, split plan: one sequence
    ("loglinear-d64-L65536", dict(B=2, H=48, L=4096)),  # level weights offset per group
    # odd L: L * num_levels is odd, so the whole problem and every group take the generic
    # path (11 heads per group)
    ("loglinear-d64-L65536", dict(B=2, H=44, L=4001)),
    # level weights 4 bytes past a 16-byte boundary: the generic path, for every group
    ("loglinear-d64-L65536", dict(B=2, H=48, L=4096, misalign=True)),
]


@pytest.mark.parametrize("name,over", HOST_CASES)
def test_host_entry_point_equals_device_path(name, over):
    """la_chunked_fwd_host (pinned host buffers in and out) returns exactly the device
    entry point's output, and that output matches the oracle on sampled rows."""
    import torch

    import chunkwise_causal_linear_gb300 as la
    over = dict(over)
    misalign = over.pop("misalign", False)
    w = workload(name, **over)
    inp = synth.make_inputs(w, seed=31)
    B, H, L, dk, dv = w["B"], w["H"], w["L"], w["dk"], w["dv"]
    lam = None
    if inp["lam"] is not None:
        flat = torch.from_numpy(inp["lam"]).reshape(-1)
        buf = torch.empty(flat.numel() + 4, dtype=torch.float32, device="cuda")
        o = 1 if misalign else 0
        buf[o:o + flat.numel()].copy_(flat)
        lam = buf[o:o + flat.numel()].view(B, H, L, -1)
        assert (lam.data_ptr() % 16 != 0) == misalign
    out_dev = la.chunked_fwd(to_device(inp["q"], w["dtype"], (B, H, L, dk)),
                             to_device(inp["k"], w["dtype"], (B, H, L, dk)),
                             to_device(inp["v"], w["dtype"], (B, H, L, dv)), C=w["C"],
                             feature_map=w["fm"], normalize=w["normalize"], level_weights=lam)
    torch.cuda.synchronize()
    out_dev = from_device(out_dev).reshape(B * H, L, dv)
    q = to_device(inp["q"], w["dtype"], (B, H, L, dk))
    k = to_device(inp["k"], w["dtype"], (B, H, L, dk))
    v = to_device(inp["v"], w["dtype"], (B, H, L, dv))
    qh, kh, vh = (x.cpu().pin_memory() for x in (q, k, v))
    outh = torch.empty((B, H, L, dv), dtype=q.dtype).pin_memory()
    qd, kd, vd = (torch.empty_like(x) for x in (q, k, v))
    od = torch.empty((B, H, L, dv), dtype=q.dtype, device="cuda")
    nl = 0 if lam is None else lam.shape[-1]
    fm = la.make_feature_map(w["fm"])
    dt = la.LA_BF16 if w["dtype"] == "bf16" else la.LA_F32
    wsb = la.la_chunked_workspace_bytes(B, H, L, dk, dv, w["C"], fm, int(w["normalize"]), nl, dt)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = la.la_chunked_fwd_host(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), outh.data_ptr(),
                                qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), od.data_ptr(), B, H, L,
                                dk, dv, w["C"], fm, int(w["normalize"]),
                                None if lam is None else lam.data_ptr(), nl, dt, ws.data_ptr(), wsb, s)
    assert rc == la.LA_OK, la.la_status_string(rc)
    torch.cuda.current_stream().synchronize()
    st = la.la_last_device_status(s)
    assert st == la.LA_OK, la.la_status_string(st)
    got = from_device(outh).reshape(B * H, L, dv)
    assert np.array_equal(got, out_dev), np.abs(got - out_dev).max()
    heads = [0, B * H - 1]
    rows = sample_rows(L, w["C"], 24, seed=31)
    ref = oracle_heads(w, inp, heads, method="scores_first", rows=rows)
    assert_close(got[heads][:, rows], ref, f"host entry point {name} {over}")
