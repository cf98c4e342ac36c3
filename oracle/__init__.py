"""CPU oracle for chunkwise causal linear attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
import this package.  The CUDA library (``chunkwise_causal_linear_gb300``) never imports
it, and this package imports nothing from there: the two share no code.  The only module
both use is ``synth`` (seeded input draws, no attention arithmetic).

The arithmetic lives in ``oracle.c`` (plain C, fp64, single-threaded per head); this
module builds it with gcc on first use, loads it with ctypes and offers numpy wrappers.
Heads are independent, so multi-head calls run one head per thread (ctypes releases the
GIL during the foreign call).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None
_lock = threading.Lock()

_dp = ctypes.POINTER(ctypes.c_double)
_lp = ctypes.POINTER(ctypes.c_long)


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (gcc -O2, IEEE arithmetic)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC,
                    "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            c_long, c_int, c_ll = ctypes.c_long, ctypes.c_int, ctypes.c_longlong
            L.orc_phi_identity.argtypes = [_dp, c_long, _dp]
            L.orc_phi_elu1.argtypes = [_dp, c_long, _dp]
            L.orc_phi_favor.argtypes = [_dp, c_long, c_int, _dp, c_int, _dp]
            L.orc_fenwick_level.argtypes = [c_long, c_long]
            L.orc_fenwick_level.restype = c_int
            L.orc_scores_first.argtypes = [_dp, _dp, _dp, c_long, c_int, c_int, c_int, c_int,
                                           _dp, c_int, _lp, c_long, _dp]
            L.orc_scores_first.restype = c_int
            L.orc_state_first.argtypes = [_dp, _dp, _dp, c_long, c_int, c_int, c_int, _dp, _dp,
                                          _dp]
            L.orc_state_recurrence.argtypes = [_dp, _dp, _dp, c_long, c_int, c_int, c_int, _dp,
                                               _dp, _dp, _dp, _dp]
            L.orc_chunked.argtypes = [_dp, _dp, _dp, c_long, c_int, c_int, c_long, c_int, c_int,
                                      _dp]
            L.orc_loglinear_recurrence.argtypes = [_dp, _dp, _dp, c_long, c_int, c_int, _dp,
                                                   c_int, c_int, _dp]
            L.orc_loglinear_recurrence.restype = c_int
            L.orc_decay_recurrence.argtypes = [_dp, _dp, _dp, c_long, c_int, c_int,
                                               ctypes.c_double, c_int, _dp]
            L.orc_decay_scores_first.argtypes = [_dp, _dp, _dp, c_long, c_int, c_int,
                                                 ctypes.c_double, c_int, _lp, c_long, _dp]
            L.orc_backward_features.argtypes = [_dp, _dp, _dp, _dp, c_long, c_int, c_int, c_int,
                                                ctypes.c_double, _dp, _dp, _dp]
            L.orc_phi_grad.argtypes = [_dp, c_long, c_int, c_int, _dp, c_int, _dp, _dp]
            L.orc_backward_features_ll.argtypes = [_dp, _dp, _dp, _dp, _dp, c_int, c_long, c_int,
                                                   c_int, c_int, _dp, _dp, _dp]
            L.orc_backward_features_ll.restype = c_int
            for name in ("orc_state_flops", "orc_score_flops", "orc_total_flops"):
                getattr(L, name).argtypes = [c_ll, c_ll, c_ll]
                getattr(L, name).restype = c_ll
            L.orc_intra_memory.argtypes = [c_ll]
            L.orc_intra_memory.restype = c_ll
            L.orc_is_full_attention.argtypes = [c_ll, c_ll]
            L.orc_is_full_attention.restype = c_int
            L.orc_is_linear.argtypes = [c_ll]
            L.orc_is_linear.restype = c_int
            L.orc_state_elems.argtypes = [c_ll, c_ll]
            L.orc_state_elems.restype = c_ll
            L.orc_kv_cache_elems.argtypes = [c_ll, c_ll]
            L.orc_kv_cache_elems.restype = c_ll
            _lib = L
    return _lib


def _c(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    return None if a is None else a.ctypes.data_as(_dp)


# ---------------------------------------------------------------------------
# feature maps
# ---------------------------------------------------------------------------
def phi(x: np.ndarray, kind: str, omega: np.ndarray | None = None) -> np.ndarray:
    """Feature map of rows x [n, d] -> [n, D] in float64 (identity / elu1 / favor)."""
    x = _c(x)
    n, d = x.shape
    if kind == "identity":
        out = np.empty_like(x)
        lib().orc_phi_identity(_p(x), x.size, _p(out))
    elif kind == "elu1":
        out = np.empty_like(x)
        lib().orc_phi_elu1(_p(x), x.size, _p(out))
    elif kind == "favor":
        om = _c(omega)
        m = om.shape[0]
        assert om.shape[1] == d
        out = np.empty((n, m), dtype=np.float64)
        lib().orc_phi_favor(_p(x), n, d, _p(om), m, _p(out))
    else:
        raise ValueError(kind)
    return out


def fenwick_level(t: int, s: int) -> int:
    return lib().orc_fenwick_level(t, s)


# ---------------------------------------------------------------------------
# single-head orders (inputs already feature-mapped: fq, fk [L, D], v [L, dv])
# ---------------------------------------------------------------------------
def scores_first(fq, fk, v, causal=True, normalize=False, lam=None, rows=None):
    fq, fk, v = _c(fq), _c(fk), _c(v)
    L, D = fq.shape
    dv = v.shape[1]
    lam_a = None if lam is None else _c(lam)
    nl = 0 if lam is None else lam_a.shape[1]
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = L if rows is None else len(rows_a)
    out = np.empty((n, dv), dtype=np.float64)
    rc = lib().orc_scores_first(_p(fq), _p(fk), _p(v), L, D, dv, int(causal), int(normalize),
                                _p(lam_a), nl,
                                None if rows_a is None else rows_a.ctypes.data_as(_lp), n,
                                _p(out))
    if rc != 0:
        raise ValueError("level weights have too few levels for this sequence length")
    return out


def state_first(fq, fk, v, normalize=False, return_state=False):
    fq, fk, v = _c(fq), _c(fk), _c(v)
    L, D = fq.shape
    dv = v.shape[1]
    out = np.empty((L, dv))
    S = np.empty((D, dv))
    z = np.empty(D)
    lib().orc_state_first(_p(fq), _p(fk), _p(v), L, D, dv, int(normalize), _p(out), _p(S), _p(z))
    return (out, S, z) if return_state else out


def state_recurrence(fq, fk, v, normalize=False, S0=None, z0=None, return_state=False):
    fq, fk, v = _c(fq), _c(fk), _c(v)
    L, D = fq.shape
    dv = v.shape[1]
    out = np.empty((L, dv))
    S = np.empty((D, dv))
    z = np.empty(D)
    S0a = None if S0 is None else _c(S0)
    z0a = None if z0 is None else _c(z0)
    lib().orc_state_recurrence(_p(fq), _p(fk), _p(v), L, D, dv, int(normalize), _p(S0a),
                               _p(z0a), _p(out), _p(S), _p(z))
    return (out, S, z) if return_state else out


def chunked(fq, fk, v, C, normalize=False, unmasked_intra=False):
    fq, fk, v = _c(fq), _c(fk), _c(v)
    L, D = fq.shape
    dv = v.shape[1]
    out = np.empty((L, dv))
    lib().orc_chunked(_p(fq), _p(fk), _p(v), L, D, dv, int(C), int(normalize),
                      int(unmasked_intra), _p(out))
    return out


def loglinear_recurrence(fq, fk, v, lam, normalize=False):
    fq, fk, v, lam = _c(fq), _c(fk), _c(v), _c(lam)
    L, D = fq.shape
    dv = v.shape[1]
    out = np.empty((L, dv))
    rc = lib().orc_loglinear_recurrence(_p(fq), _p(fk), _p(v), L, D, dv, _p(lam), lam.shape[1],
                                        int(normalize), _p(out))
    if rc != 0:
        raise ValueError("level weights have too few levels for this sequence length")
    return out


def decay_recurrence(fq, fk, v, gamma, normalize=False):
    """Retention update S_t = gamma S_{t-1} + phi(k_t) v_t^T (z decays alike)."""
    fq, fk, v = _c(fq), _c(fk), _c(v)
    L, D = fq.shape
    dv = v.shape[1]
    out = np.empty((L, dv))
    lib().orc_decay_recurrence(_p(fq), _p(fk), _p(v), L, D, dv, float(gamma), int(normalize),
                               _p(out))
    return out


def decay_scores_first(fq, fk, v, gamma, normalize=False, rows=None):
    """The decayed output as a sum over the past with weights gamma^(t-s)."""
    fq, fk, v = _c(fq), _c(fk), _c(v)
    L, D = fq.shape
    dv = v.shape[1]
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = L if rows is None else len(rows_a)
    out = np.empty((n, dv))
    lib().orc_decay_scores_first(_p(fq), _p(fk), _p(v), L, D, dv, float(gamma), int(normalize),
                                 None if rows_a is None else rows_a.ctypes.data_as(_lp), n,
                                 _p(out))
    return out


# ---------------------------------------------------------------------------
# backward pass
# ---------------------------------------------------------------------------
_FM_CODE = {"identity": 0, "elu1": 1, "favor": 2}


def backward_features(fq, fk, v, dout, normalize=False, gamma=None, lam=None):
    """Gradients (dphi(q), dphi(k), dv) of the causal output, by the chain rule on the plain
    definition (gamma: Retention decay, None for none; lam [L, NL]: the log-linear level
    weights of each query row, None for none)."""
    fq, fk, v, dout = _c(fq), _c(fk), _c(v), _c(dout)
    L, D = fq.shape
    dv = v.shape[1]
    dfq, dfk, dvo = np.empty((L, D)), np.empty((L, D)), np.empty((L, dv))
    if lam is not None:
        if gamma is not None:
            raise ValueError("the decay is defined for the plain causal mask only")
        lam = _c(lam)
        rc = lib().orc_backward_features_ll(_p(fq), _p(fk), _p(v), _p(dout), _p(lam),
                                            lam.shape[1], L, D, dv, int(normalize), _p(dfq),
                                            _p(dfk), _p(dvo))
        if rc != 0:
            raise ValueError("level weights have too few levels for this sequence length")
        return dfq, dfk, dvo
    lib().orc_backward_features(_p(fq), _p(fk), _p(v), _p(dout), L, D, dv, int(normalize),
                                -1.0 if gamma is None else float(gamma), _p(dfq), _p(dfk),
                                _p(dvo))
    return dfq, dfk, dvo


def phi_grad(x, dphi, kind, omega=None):
    """dx from dphi through the feature map (identity / elu1 / favor)."""
    x, dphi = _c(x), _c(dphi)
    rows, d = x.shape
    om = None if omega is None else _c(omega)
    m = 0 if om is None else om.shape[0]
    dx = np.empty_like(x)
    lib().orc_phi_grad(_p(x), rows, d, _FM_CODE[kind], _p(om), m, _p(dphi), _p(dx))
    return dx


def head_backward(q, k, v, dout, fm="identity", omega=None, normalize=False, gamma=None,
                  lam=None):
    """(dq, dk, dv) of one head from raw q, k [L, dk], v, dout [L, dv] (float64)."""
    fq, fk = phi(q, fm, omega), phi(k, fm, omega)
    dfq, dfk, dvo = backward_features(fq, fk, v, dout, normalize, gamma, lam)
    return phi_grad(q, dfq, fm, omega), phi_grad(k, dfk, fm, omega), dvo


def backward(q, k, v, dout, fm="identity", omega=None, normalize=False, gamma=None,
             threads=None, lam=None):
    """All heads: q, k [n, L, dk], v, dout [n, L, dv] -> (dq, dk, dv) stacked over heads
    (lam [n, L, NL]: log-linear level weights)."""
    n = q.shape[0]
    res = [None] * n

    def one(h):
        res[h] = head_backward(q[h], k[h], v[h], dout[h], fm, omega, normalize, gamma,
                               None if lam is None else lam[h])

    threads = threads or min(n, os.cpu_count() or 1)
    if threads <= 1 or n == 1:
        for h in range(n):
            one(h)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(one, range(n)))
    return tuple(np.stack([r[i] for r in res]) for i in range(3))


# ---------------------------------------------------------------------------
# cost model
# ---------------------------------------------------------------------------
def cost_model(L: int, D: int, C: int) -> dict:
    l_ = lib()
    return dict(state=l_.orc_state_flops(L, D, C), score=l_.orc_score_flops(L, D, C),
                total=l_.orc_total_flops(L, D, C), intra_memory=l_.orc_intra_memory(C),
                is_full_attention=bool(l_.orc_is_full_attention(L, C)),
                is_linear=bool(l_.orc_is_linear(C)))


def state_vs_kv(L: int, d: int) -> tuple[int, int]:
    return lib().orc_state_elems(L, d), lib().orc_kv_cache_elems(L, d)


# ---------------------------------------------------------------------------
# whole-problem helpers over heads (raw q, k, v as float64 [n_heads, L, d])
# ---------------------------------------------------------------------------
def head_forward(q, k, v, fm="identity", omega=None, normalize=False, lam=None,
                 method="recurrence", rows=None, causal=True, gamma=None):
    """One head from raw q,k,v [L, d] (float64): feature map, then the chosen order.

    method: "recurrence" (chunk size 1; log-linear uses the Fenwick recurrence) or
    "scores_first" (the definition; rows= selects output rows).  causal=False: every query
    sees every key ("attention と線形の間" section 1; the bidirectional normalised form of
    "Linear Attention / Performerの理論と実装"), computed state first.  gamma: the
    Retention decay of that page (S_t = gamma S_{t-1} + phi(k_t) v_t^T), causal only.
    """
    fq, fk = phi(q, fm, omega), phi(k, fm, omega)
    if gamma is not None:
        if lam is not None or not causal:
            raise ValueError("the decay is defined for the plain causal mask only")
        if method == "scores_first":
            return decay_scores_first(fq, fk, v, gamma, normalize=normalize, rows=rows)
        if method == "recurrence":
            out = decay_recurrence(fq, fk, v, gamma, normalize=normalize)
            return out if rows is None else out[np.asarray(rows)]
        raise ValueError(method)
    if not causal:
        if lam is not None:
            raise ValueError("the log-linear mask is causal")
        if method == "scores_first":
            return scores_first(fq, fk, v, causal=False, normalize=normalize, rows=rows)
        out = state_first(fq, fk, v, normalize=normalize)
        return out if rows is None else out[np.asarray(rows)]
    if method == "scores_first":
        return scores_first(fq, fk, v, causal=True, normalize=normalize, lam=lam, rows=rows)
    if method == "recurrence":
        if lam is not None:
            out = loglinear_recurrence(fq, fk, v, lam, normalize=normalize)
        else:
            out = state_recurrence(fq, fk, v, normalize=normalize)
        return out if rows is None else out[np.asarray(rows)]
    raise ValueError(method)


def forward(q, k, v, fm="identity", omega=None, normalize=False, lam=None,
            method="recurrence", rows=None, threads=None, causal=True, gamma=None):
    """All heads: q,k [n, L, dk], v [n, L, dv] float64 -> [n, L or len(rows), dv]."""
    n = q.shape[0]
    results = [None] * n

    def one(h):
        results[h] = head_forward(q[h], k[h], v[h], fm, omega, normalize,
                                  None if lam is None else lam[h], method, rows, causal, gamma)

    threads = threads or min(n, os.cpu_count() or 1)
    if threads <= 1 or n == 1:
        for h in range(n):
            one(h)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(one, range(n)))
    return np.stack(results)
