"""Seeded synthetic inputs for chunkwise causal linear attention.

This module is shared by the CPU oracle tests and by the CUDA path's tests and
benchmark. It draws random numbers and rounds them to the storage dtype; it holds
none of the attention arithmetic (no feature map, no score, no state, no mask).

Every tensor is generated per (b, h) head from a counter-based generator (numpy's
Philox keyed by ``(seed, tensor id, head)``), so any subset of heads can be
regenerated on its own -- the oracle side draws only the heads it samples, the GPU
side draws all of them, and both see identical values.

Workload recipes (shapes and distributions) are the five workloads the library is
measured on; see ``WORKLOADS``.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

# tensor ids used in the Philox key
T_Q, T_K, T_V, T_LAMBDA, T_OMEGA_G, T_OMEGA_CHI, T_DOUT = 1, 2, 3, 4, 5, 6, 7


def _gen(seed: int, tensor: int, head: int) -> np.random.Generator:
    key = np.array([seed & 0xFFFFFFFFFFFFFFFF, (tensor << 40) | (head & 0xFFFFFFFFFF)],
                   dtype=np.uint64)
    return np.random.Generator(np.random.Philox(key=key))


# ---------------------------------------------------------------------------
# bf16 storage (round-to-nearest-even), kept as raw uint16 bit patterns
# ---------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (RNE) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------------------
# per-head draws
# ---------------------------------------------------------------------------
def head_values(seed: int, tensor: int, head: int, L: int, d: int, dist: str, scale: float,
                dtype: str) -> np.ndarray:
    """One head's [L, d] tensor as stored: uint16 bf16 bits, or float32.

    dist: "normal" (N(0,1) * scale), "uniform01" (U[0,1)), "int" (integers uniform in
    {-scale..scale}, e.g. scale=3 gives {-3..3}).
    """
    g = _gen(seed, tensor, head)
    if dist == "normal":
        x = g.standard_normal((L, d), dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
    elif dist == "uniform01":
        x = g.random((L, d), dtype=np.float32)
    elif dist == "int":
        r = int(scale)
        x = g.integers(-r, r + 1, size=(L, d)).astype(np.float32)
    else:
        raise ValueError(dist)
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    if dtype == "f32":
        return x
    raise ValueError(dtype)


def tensor_values(seed: int, tensor: int, B: int, H: int, L: int, d: int, dist: str,
                  scale: float, dtype: str, heads=None, threads: int | None = None) -> np.ndarray:
    """[n_heads, L, d] for the listed heads (default: all B*H heads, b-major)."""
    heads = list(range(B * H)) if heads is None else list(heads)
    out = np.empty((len(heads), L, d), dtype=np.uint16 if dtype == "bf16" else np.float32)

    def one(i):
        out[i] = head_values(seed, tensor, heads[i], L, d, dist, scale, dtype)

    threads = threads or min(len(heads), os.cpu_count() or 1, 32)
    if threads <= 1 or len(heads) <= 1:
        for i in range(len(heads)):
            one(i)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(one, range(len(heads))))
    return out


def block_orthogonal_gaussian(seed: int, m: int, d: int) -> np.ndarray:
    """[m, d] float32 random matrix drawn the way the Performer page draws its orthogonal
    random features: ceil(m/d) independent d x d Gaussian matrices, each replaced by the
    orthogonal factor of its QR decomposition, each row rescaled to the norm of a
    chi(d)-distributed sample (sqrt of a chi-square with d degrees of freedom), stacked
    and cut to m rows.  Page: "Linear Attention / Performerの理論と実装", section
    "直交ランダム特徴量" and its create_orthogonal_random_matrix implementation.

    The feature map consumes this matrix as data; how it was drawn does not enter the
    attention arithmetic (QR sign conventions, RNG) -- both sides receive the same array.
    """
    nb = (m + d - 1) // d
    blocks = []
    for b in range(nb):
        g = _gen(seed, T_OMEGA_G, b)
        G = g.standard_normal((d, d))
        Qm, _ = np.linalg.qr(G)
        chi = np.sqrt(_gen(seed, T_OMEGA_CHI, b).chisquare(d, size=d))
        blocks.append(chi[:, None] * Qm)
    return np.vstack(blocks)[:m].astype(np.float32)


def iid_gaussian(seed: int, m: int, d: int) -> np.ndarray:
    """[m, d] float64 i.i.d. N(0,1) rows (used for the unbiasedness check of FAVOR+)."""
    return _gen(seed, T_OMEGA_G, 1 << 30).standard_normal((m, d))


# ---------------------------------------------------------------------------
# the measured workloads
# ---------------------------------------------------------------------------
WORKLOADS = {
    # exactness case: integers in {-3..3} stored as fp32, identity features, no normaliser
    "tiny-int-exact": dict(B=1, H=1, L=64, dk=16, dv=16, dtype="f32", dist="int", scale=3.0,
                           fm="identity", m=0, normalize=False, C=64, Cs=(1, 4, 16, 64),
                           loglinear=False),
    # unnormalised identity-feature causal linear attention, q,k,v ~ N(0,1)/sqrt(64)
    "identity-d64-L2048": dict(B=4, H=8, L=2048, dk=64, dv=64, dtype="bf16", dist="normal",
                               scale=1.0 / 8.0, fm="identity", m=0, normalize=False, C=64,
                               Cs=(64,), loglinear=False),
    # elu+1 features with the normaliser, q,k,v ~ N(0,1)
    "elu1-norm-d128-L8192": dict(B=8, H=16, L=8192, dk=128, dv=128, dtype="bf16",
                                 dist="normal", scale=1.0, fm="elu1", m=0, normalize=True,
                                 C=64, Cs=(16, 32, 64, 128, 256), loglinear=False),
    # FAVOR+ positive random features, m=256 from d=64, with the normaliser
    "favor-m256-d64-L16384": dict(B=2, H=12, L=16384, dk=64, dv=64, dtype="bf16",
                                  dist="normal", scale=1.0, fm="favor", m=256, normalize=True,
                                  C=64, Cs=(64,), loglinear=False),
    # the elu+1 normalised workload with the Retention decay, gamma = 0.98 (the scalar gate
    # value printed in the Kimi/Qwen comparison page, section 3.3.7)
    "decay-elu1-norm-d128-L8192": dict(B=8, H=16, L=8192, dk=128, dv=128, dtype="bf16",
                                       dist="normal", scale=1.0, fm="elu1", m=0,
                                       normalize=True, C=64, Cs=(64,), loglinear=False,
                                       gamma=0.98),
    # Fenwick-level-weighted log-linear mask, 17 level weights per token ~ U(0,1)
    "loglinear-d64-L65536": dict(B=1, H=16, L=65536, dk=64, dv=64, dtype="bf16",
                                 dist="normal", scale=1.0 / 8.0, fm="identity", m=0,
                                 normalize=False, C=64, Cs=(64,), loglinear=True),
}


def num_levels(L: int) -> int:
    """Number of Fenwick levels a sequence of length L can use: level 0 (the token
    itself) plus 1 + floor(log2(t XOR s)) for s < t < L, i.e. 1 + ceil(log2(L))."""
    return 1 + max(1, math.ceil(math.log2(max(L, 2))))


def make_inputs(w: dict, seed: int, heads=None, with_omega: bool = True) -> dict:
    """Draw q, k, v (and lambda, omega where the workload has them) for the listed heads.

    Returns numpy arrays: q,k,v [n, L, d] (uint16 bf16 bits or float32), lam [n, L, NL]
    float32 or None, omega [m, dk] float32 or None.
    """
    B, H, L = w["B"], w["H"], w["L"]
    q = tensor_values(seed, T_Q, B, H, L, w["dk"], w["dist"], w["scale"], w["dtype"], heads)
    k = tensor_values(seed, T_K, B, H, L, w["dk"], w["dist"], w["scale"], w["dtype"], heads)
    v = tensor_values(seed, T_V, B, H, L, w["dv"], w["dist"], w["scale"], w["dtype"], heads)
    lam = None
    if w.get("loglinear"):
        lam = tensor_values(seed, T_LAMBDA, B, H, L, num_levels(L), "uniform01", 1.0, "f32",
                            heads)
    omega = None
    if w["fm"] == "favor" and with_omega:
        omega = block_orthogonal_gaussian(seed, w["m"], w["dk"])
    return dict(q=q, k=k, v=v, lam=lam, omega=omega)


def as_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Stored values as float64 (exact: every bf16 and fp32 value is a double)."""
    if dtype == "bf16":
        return bf16_bits_to_f32(x).astype(np.float64)
    return np.asarray(x, dtype=np.float64)
