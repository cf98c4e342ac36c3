"""Shared helpers of the GPU parity tests: draw seeded inputs, run the library through
its C ABI, run the oracle on the same values, compare."""
from __future__ import annotations

import numpy as np

import synth

# bf16 tolerance: max |err| <= 2e-2 * max |ref| and ||err|| / ||ref|| <= 5e-3 (relative RMS)
MAX_ABS_FRAC = 2e-2
REL_RMS = 5e-3


def to_device(x: np.ndarray, dtype: str, shape):
    import torch
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.reshape(shape).cuda()


def from_device(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def workload(base: str, **over) -> dict:
    w = dict(synth.WORKLOADS[base])
    w.update(over)
    return w


def run_gpu(w: dict, inp: dict, C: int, path: int = 0):
    """Runs the library on all heads of inp; returns (out float64 [B*H, L, dv], torch out)."""
    import torch

    import chunkwise_causal_linear_gb300 as la
    B, H, L, dk, dv = w["B"], w["H"], w["L"], w["dk"], w["dv"]
    q = to_device(inp["q"], w["dtype"], (B, H, L, dk))
    k = to_device(inp["k"], w["dtype"], (B, H, L, dk))
    v = to_device(inp["v"], w["dtype"], (B, H, L, dv))
    omega = None if inp["omega"] is None else torch.from_numpy(inp["omega"]).cuda()
    lam = None if inp["lam"] is None else torch.from_numpy(inp["lam"]).reshape(
        B, H, L, -1).cuda()
    out = la.chunked_fwd(q, k, v, C=C, feature_map=w["fm"], omega=omega,
                         normalize=w["normalize"], level_weights=lam, path=path)
    torch.cuda.synchronize()
    st = la.la_last_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == la.LA_OK, la.la_status_string(st)
    return from_device(out).reshape(B * H, L, dv), out


def oracle_heads(w: dict, inp: dict, heads_idx, method="recurrence", rows=None):
    """Oracle output for the given positions in inp's head axis."""
    import oracle
    q = synth.as_f64(inp["q"][heads_idx], w["dtype"])
    k = synth.as_f64(inp["k"][heads_idx], w["dtype"])
    v = synth.as_f64(inp["v"][heads_idx], w["dtype"])
    lam = None if inp["lam"] is None else inp["lam"][heads_idx].astype(np.float64)
    om = None if inp["omega"] is None else inp["omega"].astype(np.float64)
    return oracle.forward(q, k, v, fm=w["fm"], omega=om, normalize=w["normalize"], lam=lam,
                          method=method, rows=rows)


def errors(out: np.ndarray, ref: np.ndarray) -> dict:
    err = out - ref
    return dict(max_abs=float(np.abs(err).max()), max_ref=float(np.abs(ref).max()),
                rel_rms=float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300)))


def assert_close(out: np.ndarray, ref: np.ndarray, what=""):
    assert np.isfinite(out).all(), f"{what}: non-finite output"
    e = errors(out, ref)
    assert e["max_abs"] <= MAX_ABS_FRAC * e["max_ref"], f"{what}: {e}"
    assert e["rel_rms"] <= REL_RMS, f"{what}: {e}"
    return e


def sample_rows(L: int, C: int, n_random: int, seed: int):
    """First and last 2C rows of a head plus random rows in between (sorted, unique)."""
    rng = np.random.default_rng(seed)
    edge = list(range(min(L, 2 * C))) + list(range(max(0, L - 2 * C), L))
    mid = rng.integers(0, L, size=n_random).tolist() if L > 0 else []
    return np.array(sorted(set(edge + mid)), dtype=np.int64)
