"""Host-side checks of the C ABI: no GPU needed, nothing is launched.

The library must build for sm_103a, load, and export every function include/la_chunked.h
declares; argument errors must come back as status codes before any device work.
"""
import ctypes
import os
import re

import pytest

import chunkwise_causal_linear_gb300 as la
from chunkwise_causal_linear_gb300 import build as la_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    la_build.build()
    return la.lib()


def header_functions():
    txt = open(os.path.join(ROOT, "include", "la_chunked.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(la_[a-z_0-9]+)\s*\(", txt)))


def test_header_declares_the_binding_exports():
    assert sorted(la.EXPORTS) == header_functions()


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
    assert la.la_version() == "0.1.0"


def test_status_strings(lib):
    for s in (la.LA_OK, la.LA_ERR_NULL, la.LA_ERR_SHAPE, la.LA_ERR_UNSUPPORTED,
              la.LA_ERR_WORKSPACE, la.LA_ERR_CUDA, la.LA_ERR_TIMEOUT, la.LA_ERR_DEVICE):
        assert la.la_status_string(s) and la.la_status_string(s) != "unknown status"
    assert la.la_status_string(12345) == "unknown status"


def test_cost_model_matches_printed_table(lib, golden):
    for C, state, score, total, _ in golden("chunked_cost_model_L1024_d64.txt"):
        st, sc = la.la_cost_model(1024, 64, int(C))
        assert (st, sc, st + sc) == (int(state), int(score), int(total))
    with pytest.raises(la.LAError):
        la.la_cost_model(-1, 64, 64)


FAKE = 1 << 20  # a non-NULL value: argument checks must fail before it is ever used


def call(q=FAKE, k=FAKE, v=FAKE, out=FAKE, B=1, H=1, L=64, dk=16, dv=16, C=16, fm=None,
         normalize=0, lam=None, nl=0, dtype=la.LA_F32, ws=None, wsb=0, path=la.LA_PATH_AUTO):
    return la.la_chunked_fwd_path(q, k, v, out, B, H, L, dk, dv, C, fm, normalize, lam, nl,
                                  dtype, ws, wsb, None, path)


def test_null_pointers_rejected(lib):
    assert call(q=None) == la.LA_ERR_NULL
    assert call(k=None) == la.LA_ERR_NULL
    assert call(v=None) == la.LA_ERR_NULL
    assert call(out=None) == la.LA_ERR_NULL
    # FAVOR+ without omega
    assert call(fm=la.make_feature_map("favor", 64, 0), dtype=la.LA_BF16) == la.LA_ERR_NULL
    assert la.la_chunked_fwd_host(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 4, 4,
                                  4, None, 0, None, 0, la.LA_F32, None, 0, None) == la.LA_ERR_NULL


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=-1), dict(L=0), dict(dk=0), dict(dv=-3)])
def test_bad_shapes_rejected(lib, kw):
    assert call(**kw) == la.LA_ERR_SHAPE


def test_unsupported_combinations_rejected(lib):
    assert call(dtype=7) == la.LA_ERR_UNSUPPORTED
    assert call(fm=la.make_feature_map(9)) == la.LA_ERR_UNSUPPORTED
    assert call(dk=1024) == la.LA_ERR_UNSUPPORTED
    # log-linear needs a power-of-two chunk size once there is more than one chunk
    assert call(lam=FAKE, nl=7, C=24) == la.LA_ERR_UNSUPPORTED
    # ...and enough levels for L
    assert call(lam=FAKE, nl=6, C=16) == la.LA_ERR_SHAPE
    assert call(fm=la.make_feature_map("favor", 0, FAKE)) == la.LA_ERR_SHAPE


def test_plan_simt_grid_and_clamping(lib):
    fm = la.make_feature_map("identity")
    rc, info = la.la_chunked_plan(2, 3, 100, 16, 40, 0, fm, 0, 0, 0, la.LA_F32,
                                  la.LA_PATH_SIMT, 152)
    assert rc == la.LA_OK
    assert info["path"] == la.LA_PATH_SIMT and info["chunk"] == 1 and info["n_chunks"] == 100
    assert (info["grid_x"], info["grid_y"]) == (6, 2)
    rc, info = la.la_chunked_plan(1, 1, 100, 16, 16, 1000, fm, 0, 0, 0, la.LA_F32,
                                  la.LA_PATH_SIMT, 152)
    assert info["chunk"] == 100 and info["n_chunks"] == 1
    assert info["workspace_bytes"] == 0


def test_plan_loglinear_workspace(lib):
    fm = la.make_feature_map("identity")
    # L = 65536, C = 64: 1024 chunks -> 10 inter-chunk level states per (head, slice)
    rc, info = la.la_chunked_plan(1, 16, 65536, 64, 64, 64, fm, 0, 1, 17, la.LA_BF16,
                                  la.LA_PATH_SIMT, 152)
    assert rc == la.LA_OK
    assert info["workspace_bytes"] == 16 * 2 * 10 * (64 * 32 + 64) * 4
    # one chunk: no inter-chunk levels, no workspace, any C
    rc, info = la.la_chunked_plan(1, 1, 50, 8, 8, 50, fm, 0, 1, 7, la.LA_F32, la.LA_PATH_SIMT,
                                  152)
    assert rc == la.LA_OK and info["workspace_bytes"] == 0


def test_workspace_too_small_rejected_before_launch(lib):
    # the workspace check needs the device's SM count; on a machine without a GPU the
    # call reports the CUDA failure instead -- either way nothing runs
    rc = call(lam=FAKE, nl=7, C=16, L=64)
    assert rc in (la.LA_ERR_WORKSPACE, la.LA_ERR_CUDA)


# ---------------------------------------------------------------------------
# decoding step: host-side checks (nothing launched)
# ---------------------------------------------------------------------------
def test_decode_state_elems(lib):
    fm = la.make_feature_map("identity")
    assert la.la_decode_state_elems(2, 3, 64, 32, fm, 0) == (2 * 3 * 64 * 32, 2 * 3 * 64)
    # log-linear: num_levels - 1 level states
    assert la.la_decode_state_elems(2, 3, 64, 32, fm, 17) == (2 * 3 * 16 * 64 * 32, 2 * 3 * 16 * 64)
    fav = la.make_feature_map("favor", 256, 1)
    assert la.la_decode_state_elems(1, 2, 64, 64, fav, 0) == (2 * 256 * 64, 2 * 256)
    assert la.la_decode_state_elems(0, 2, 64, 64, fm, 0) == (0, 0)


def test_decode_rejects_bad_arguments_before_launch(lib):
    fm = la.make_feature_map("identity")
    ok = ctypes.c_void_p(16)  # never dereferenced: every call below fails on the host
    args = dict(B=1, H=1, dk=8, dv=8, feature_map=fm, normalize=0, level_weights=None,
                num_levels=0, t=0, dtype=la.LA_F32, stream=None)
    assert la.la_decode_step(None, ok, ok, ok, ok, None, **args) == la.LA_ERR_NULL
    assert la.la_decode_step(ok, ok, ok, ok, None, None, **args) == la.LA_ERR_NULL
    # the normaliser needs its state
    assert la.la_decode_step(ok, ok, ok, ok, ok, None, **dict(args, normalize=1)) == la.LA_ERR_NULL
    assert la.la_decode_step(ok, ok, ok, ok, ok, None, **dict(args, dk=0)) == la.LA_ERR_SHAPE
    # level weights: position t+1 = 8 needs level 4 (trailing zeros 3), i.e. num_levels >= 5
    ll = dict(args, level_weights=ok, num_levels=4, t=7)
    assert la.la_decode_step(ok, ok, ok, ok, ok, None, **ll) == la.LA_ERR_SHAPE
    assert la.la_decode_step(ok, ok, ok, ok, ok, None, **dict(ll, t=-1)) == la.LA_ERR_SHAPE
    # FAVOR+ needs omega
    fav = la.make_feature_map("favor", 16, 0)
    assert la.la_decode_step(ok, ok, ok, ok, ok, None, **dict(args, feature_map=fav)) == la.LA_ERR_NULL
    assert la.la_decode_step(ok, ok, ok, ok, ok, None, **dict(args, dtype=7)) == la.LA_ERR_UNSUPPORTED


def test_noncausal_workspace_and_errors(lib):
    fm = la.make_feature_map("identity")
    assert la.la_noncausal_workspace_bytes(2, 3, 100, 64, 32, fm, 1, la.LA_BF16) >= 2 * 3 * (64 * 32 + 64) * 4
    # D above 256 is not covered
    assert la.la_noncausal_workspace_bytes(1, 1, 100, 300, 32, fm, 1, la.LA_F32) == 0
    ok = ctypes.c_void_p(16)
    assert la.la_noncausal_fwd(None, ok, ok, ok, 1, 1, 8, 8, 8, fm, 0, la.LA_F32, ok, 1 << 20,
                               None) == la.LA_ERR_NULL
    assert la.la_noncausal_fwd(ok, ok, ok, ok, 1, 1, 8, 8, 8, fm, 0, la.LA_F32, None, 0,
                               None) in (la.LA_ERR_WORKSPACE, la.LA_ERR_CUDA)


def test_decay_arguments_and_plan(lib):
    fm = la.make_feature_map("elu1")
    ok = ctypes.c_void_p(16)
    for g in (0.0, -1.0, 1.0001, float("nan"), float("inf")):
        assert la.la_decay_fwd(ok, ok, ok, ok, 1, 1, 256, 64, 64, 64, fm, 1, g, la.LA_BF16, None,
                               0, None, la.LA_PATH_AUTO) == la.LA_ERR_ARG, g
        assert la.la_decay_workspace_bytes(1, 1, 256, 64, 64, 64, fm, 1, g, la.LA_BF16) == 0
        assert la.la_decay_decode_step(ok, ok, ok, ok, ok, ok, 1, 1, 64, 64, fm, 1, g,
                                       la.LA_BF16, None) == la.LA_ERR_ARG, g
    assert la.la_decay_fwd(None, ok, ok, ok, 1, 1, 256, 64, 64, 64, fm, 1, 0.9, la.LA_BF16,
                           None, 0, None, 0) == la.LA_ERR_NULL
    assert la.la_decay_decode_step(ok, ok, ok, ok, ok, None, 1, 1, 64, 64, fm, 1, 0.9,
                                   la.LA_BF16, None) == la.LA_ERR_NULL
    # tensor cores: C = 64 and gamma >= 0.5 only; the generic path takes the rest
    rc, info = la.la_decay_plan(8, 16, 8192, 128, 128, 64, fm, 1, 0.98, la.LA_BF16,
                                la.LA_PATH_AUTO, 152)
    assert rc == la.LA_OK and info["path"] == la.LA_PATH_TC
    for C, g in ((64, 0.49), (32, 0.98), (128, 0.98)):
        rc, info = la.la_decay_plan(8, 16, 8192, 128, 128, C, fm, 1, g, la.LA_BF16,
                                    la.LA_PATH_AUTO, 152)
        assert rc == la.LA_OK and info["path"] == la.LA_PATH_SIMT, (C, g)
        rc, _ = la.la_decay_plan(8, 16, 8192, 128, 128, C, fm, 1, g, la.LA_BF16, la.LA_PATH_TC,
                                 152)
        assert rc == la.LA_ERR_UNSUPPORTED
    # few heads: the sequence split's totals need a workspace, as for the plain mask
    rc, info = la.la_decay_plan(1, 1, 8192, 128, 128, 64, fm, 1, 0.98, la.LA_BF16,
                                la.LA_PATH_AUTO, 152)
    assert rc == la.LA_OK and info["n_launches"] == 2 and info["workspace_bytes"] > 0
    assert la.la_status_string(la.LA_ERR_ARG) != "unknown status"


def test_backward_workspace_and_errors(lib):
    fm = la.make_feature_map("elu1")
    rows = 2 * 3 * 100
    need = la.la_chunked_bwd_workspace_bytes(2, 3, 100, 64, 32, 64, fm, 1, la.LA_BF16)
    # phi(q), phi(k), dphi(q), dphi(k) [D], [num, den], D', v' [dv + 1], D, dv [dv]
    assert need >= rows * 4 * (4 * 64 + 3 * 33 + 2 * 32)
    assert la.la_chunked_bwd_workspace_bytes(1, 1, 100, 600, 32, 64, fm, 1, la.LA_F32) == 0
    ok = ctypes.c_void_p(16)
    args = (1, 1, 64, 16, 16, 64, fm)
    assert la.la_chunked_bwd(None, ok, ok, ok, ok, ok, ok, *args, 0, 1.0, la.LA_F32, ok,
                             1 << 20, None) == la.LA_ERR_NULL
    assert la.la_chunked_bwd(ok, ok, ok, None, ok, ok, ok, *args, 1, 1.0, la.LA_F32, ok,
                             1 << 20, None) == la.LA_ERR_NULL
    assert la.la_chunked_bwd(ok, ok, ok, ok, ok, ok, ok, *args, 0, 0.0, la.LA_F32, ok,
                             1 << 20, None) == la.LA_ERR_ARG
    # the workspace size depends on the device's SM count: without a GPU the call reports
    # the CUDA failure instead -- either way nothing runs
    assert la.la_chunked_bwd(ok, ok, ok, ok, ok, ok, ok, *args, 0, 1.0, la.LA_F32, ok,
                             16, None) in (la.LA_ERR_WORKSPACE, la.LA_ERR_CUDA)


def test_generic_fallback_warns_on_large_bf16_problems(monkeypatch):
    """The binding names the slow generic path when the automatic plan picks it for a large
    bf16 problem (the plan query is host-only here: a fixed SM count)."""
    import warnings

    import chunkwise_causal_linear_gb300 as la
    real_plan = la.la_chunked_plan
    monkeypatch.setattr(la, "la_chunked_plan",
                        lambda *a: real_plan(*a[:-1], 152))
    fm = la.make_feature_map("elu1")
    with warnings.catch_warnings(record=True) as rec:
        warnings.simplefilter("always")
        # d = 96 is outside the tensor-core coverage
        la._warn_if_generic(8, 16, 8192, 96, 96, 64, fm, 1, 0, la.LA_BF16, la.LA_PATH_AUTO)
        # the headline shape is covered: no warning
        la._warn_if_generic(8, 16, 8192, 128, 128, 64, fm, 1, 0, la.LA_BF16, la.LA_PATH_AUTO)
    assert len(rec) == 1 and "generic" in str(rec[0].message)
