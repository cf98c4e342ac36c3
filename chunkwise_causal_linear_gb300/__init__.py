"""Python binding of liblachunked -- chunkwise-parallel causal linear attention on GB300.

Argument marshalling only: every step of the forward pass runs in the library's CUDA
kernels.  The functions named ``la_*`` mirror the C ABI in ``include/la_chunked.h`` one to
one (pointers are passed as integers).  ``chunked_fwd`` is a convenience wrapper taking
torch tensors; torch provides the device memory and the stream, nothing else.

There is no fallback: if ``liblachunked.so`` is missing or fails to load, every call
raises.  Build it with ``python -m chunkwise_causal_linear_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblachunked.so")

LA_OK = 0
LA_ERR_NULL = -1
LA_ERR_SHAPE = -2
LA_ERR_UNSUPPORTED = -3
LA_ERR_WORKSPACE = -4
LA_ERR_CUDA = -5
LA_ERR_TIMEOUT = -6
LA_ERR_DEVICE = -7
LA_ERR_SCRATCH_LIMIT = -8
LA_ERR_ARG = -9

LA_FM_IDENTITY, LA_FM_ELU1, LA_FM_FAVOR = 0, 1, 2
LA_BF16, LA_F32 = 0, 1
LA_PATH_AUTO, LA_PATH_SIMT, LA_PATH_TC = 0, 1, 2

FEATURE_MAPS = {"identity": LA_FM_IDENTITY, "elu1": LA_FM_ELU1, "favor": LA_FM_FAVOR}

# every function the header declares (checked by the tests against include/la_chunked.h)
EXPORTS = ("la_chunked_fwd", "la_chunked_fwd_path", "la_chunked_fwd_host",
           "la_chunked_fwd_noalloc", "la_chunked_workspace_bytes", "la_chunked_plan",
           "la_last_device_status", "la_status_string", "la_cost_model", "la_decode_step",
           "la_decode_state_elems", "la_noncausal_fwd", "la_noncausal_workspace_bytes",
           "la_decay_fwd", "la_decay_decode_step", "la_decay_workspace_bytes", "la_decay_plan",
           "la_chunked_bwd", "la_chunked_bwd_workspace_bytes", "la_chunked_bwd_ll",
           "la_chunked_bwd_ll_workspace_bytes", "la_chunked_state",
           "la_state_combine", "la_chunked_fwd_init", "la_version")


class la_feature_map(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("m", ctypes.c_int), ("omega", ctypes.c_void_p)]


class la_plan_info(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("chunk", ctypes.c_int), ("n_chunks", ctypes.c_int),
                ("feature_dim", ctypes.c_int), ("grid_x", ctypes.c_int),
                ("grid_y", ctypes.c_int), ("block", ctypes.c_int),
                ("smem_bytes", ctypes.c_int), ("n_launches", ctypes.c_int),
                ("workspace_bytes", ctypes.c_size_t)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class LAError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {la_status_string(status)} ({status})" if what else
                         f"{la_status_string(status)} ({status})")


_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it is missing: there is no fallback path)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing; build it with "
                    "`python -m chunkwise_causal_linear_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            i, p, sz, ll = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_longlong
            fmp = ctypes.POINTER(la_feature_map)
            common = [i, i, i, i, i, i, fmp, i, p, i, i, p, sz, p]
            L.la_chunked_fwd.argtypes = [p, p, p, p, *common]
            L.la_chunked_fwd.restype = i
            L.la_chunked_fwd_path.argtypes = [p, p, p, p, *common, i]
            L.la_chunked_fwd_path.restype = i
            L.la_chunked_fwd_host.argtypes = [p, p, p, p, p, p, p, p, *common]
            L.la_chunked_fwd_host.restype = i
            L.la_chunked_fwd_noalloc.argtypes = [p, p, p, p, i, i, i, i, i, i, fmp, i, p, i, i, p]
            L.la_chunked_fwd_noalloc.restype = i
            L.la_chunked_workspace_bytes.argtypes = [i, i, i, i, i, i, fmp, i, i, i]
            L.la_chunked_workspace_bytes.restype = sz
            L.la_chunked_plan.argtypes = [i, i, i, i, i, i, fmp, i, i, i, i, i, i,
                                          ctypes.POINTER(la_plan_info)]
            L.la_chunked_plan.restype = i
            L.la_last_device_status.argtypes = [p]
            L.la_last_device_status.restype = i
            L.la_status_string.argtypes = [i]
            L.la_status_string.restype = ctypes.c_char_p
            L.la_cost_model.argtypes = [ll, ll, ll, ctypes.POINTER(ll), ctypes.POINTER(ll)]
            L.la_cost_model.restype = i
            L.la_decode_step.argtypes = [p, p, p, p, p, p, i, i, i, i, fmp, i, p, i, ll, i, p]
            L.la_decode_step.restype = i
            L.la_decode_state_elems.argtypes = [i, i, i, i, fmp, i, ctypes.POINTER(ll)]
            L.la_decode_state_elems.restype = ll
            L.la_noncausal_fwd.argtypes = [p, p, p, p, i, i, i, i, i, fmp, i, i, p, sz, p]
            L.la_noncausal_fwd.restype = i
            L.la_noncausal_workspace_bytes.argtypes = [i, i, i, i, i, fmp, i, i]
            L.la_noncausal_workspace_bytes.restype = sz
            f = ctypes.c_float
            L.la_decay_fwd.argtypes = [p, p, p, p, i, i, i, i, i, i, fmp, i, f, i, p, sz, p, i]
            L.la_decay_fwd.restype = i
            L.la_decay_decode_step.argtypes = [p, p, p, p, p, p, i, i, i, i, fmp, i, f, i, p]
            L.la_decay_decode_step.restype = i
            L.la_decay_workspace_bytes.argtypes = [i, i, i, i, i, i, fmp, i, f, i]
            L.la_decay_workspace_bytes.restype = sz
            L.la_decay_plan.argtypes = [i, i, i, i, i, i, fmp, i, f, i, i, i,
                                        ctypes.POINTER(la_plan_info)]
            L.la_decay_plan.restype = i
            L.la_chunked_bwd.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, i, fmp, i, f, i, p, sz,
                                         p, i]
            L.la_chunked_bwd.restype = i
            L.la_chunked_bwd_workspace_bytes.argtypes = [i, i, i, i, i, i, fmp, i, i]
            L.la_chunked_bwd_workspace_bytes.restype = sz
            L.la_chunked_bwd_ll.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, i, fmp, i, p, i, i,
                                            p, sz, p, i]
            L.la_chunked_bwd_ll.restype = i
            L.la_chunked_bwd_ll_workspace_bytes.argtypes = [i, i, i, i, i, i, fmp, i, i, i]
            L.la_chunked_bwd_ll_workspace_bytes.restype = sz
            L.la_chunked_state.argtypes = [p, p, p, p, i, i, i, i, i, fmp, f, i, p]
            L.la_chunked_state.restype = i
            L.la_state_combine.argtypes = [p, p, p, p, i, i, i, i, f, p]
            L.la_state_combine.restype = i
            L.la_chunked_fwd_init.argtypes = [p, p, p, p, i, i, i, i, i, i, fmp, i, f, p, p, i, p, sz,
                                              p, i]
            L.la_chunked_fwd_init.restype = i
            L.la_version.argtypes = []
            L.la_version.restype = ctypes.c_char_p
            _lib = L
    return _lib


def make_feature_map(kind="identity", m=0, omega_ptr=0) -> la_feature_map:
    if isinstance(kind, str):
        kind = FEATURE_MAPS[kind]
    return la_feature_map(int(kind), int(m), ctypes.c_void_p(int(omega_ptr) or None))


def _fm(fm):
    return None if fm is None else ctypes.byref(fm)


# ---- one-to-one wrappers of the C ABI ------------------------------------------------
def la_chunked_fwd(q, k, v, out, B, H, L, dk, dv, C, feature_map, normalize, level_weights,
                   num_levels, dtype, workspace, workspace_bytes, stream) -> int:
    return lib().la_chunked_fwd(q, k, v, out, B, H, L, dk, dv, C, _fm(feature_map), normalize,
                                level_weights, num_levels, dtype, workspace, workspace_bytes,
                                stream)


def la_chunked_fwd_path(q, k, v, out, B, H, L, dk, dv, C, feature_map, normalize,
                        level_weights, num_levels, dtype, workspace, workspace_bytes, stream,
                        path) -> int:
    return lib().la_chunked_fwd_path(q, k, v, out, B, H, L, dk, dv, C, _fm(feature_map),
                                     normalize, level_weights, num_levels, dtype, workspace,
                                     workspace_bytes, stream, path)


def la_chunked_fwd_host(q_host, k_host, v_host, out_host, q_dev, k_dev, v_dev, out_dev, B, H,
                        L, dk, dv, C, feature_map, normalize, level_weights, num_levels, dtype,
                        workspace, workspace_bytes, stream) -> int:
    return lib().la_chunked_fwd_host(q_host, k_host, v_host, out_host, q_dev, k_dev, v_dev,
                                     out_dev, B, H, L, dk, dv, C, _fm(feature_map), normalize,
                                     level_weights, num_levels, dtype, workspace,
                                     workspace_bytes, stream)


def la_chunked_fwd_noalloc(q, k, v, out, B, H, L, dk, dv, C, feature_map, normalize,
                           level_weights, num_levels, dtype, stream) -> int:
    """Forward pass that allocates nothing (for callers that cannot allocate device
    memory); scratch, where needed, comes from a fixed 8 MiB buffer inside the library.
    Calls that may overlap on the GPU must be serialised by the caller."""
    return lib().la_chunked_fwd_noalloc(q, k, v, out, B, H, L, dk, dv, C, _fm(feature_map),
                                        normalize, level_weights, num_levels, dtype, stream)


def la_chunked_workspace_bytes(B, H, L, dk, dv, C, feature_map, normalize, num_levels,
                               dtype) -> int:
    return lib().la_chunked_workspace_bytes(B, H, L, dk, dv, C, _fm(feature_map), normalize,
                                            num_levels, dtype)


def la_chunked_plan(B, H, L, dk, dv, C, feature_map, normalize, loglinear, num_levels, dtype,
                    path=LA_PATH_AUTO, num_sms=0):
    info = la_plan_info()
    rc = lib().la_chunked_plan(B, H, L, dk, dv, C, _fm(feature_map), normalize, loglinear,
                               num_levels, dtype, path, num_sms, ctypes.byref(info))
    return rc, info.as_dict()


def la_last_device_status(stream=0) -> int:
    return lib().la_last_device_status(stream)


def la_status_string(status: int) -> str:
    return lib().la_status_string(status).decode()


def la_cost_model(L, D, C):
    st, sc = ctypes.c_longlong(), ctypes.c_longlong()
    rc = lib().la_cost_model(L, D, C, ctypes.byref(st), ctypes.byref(sc))
    if rc != LA_OK:
        raise LAError(rc, "la_cost_model")
    return st.value, sc.value


def la_decode_step(q, k, v, out, state, zstate, B, H, dk, dv, feature_map, normalize,
                   level_weights, num_levels, t, dtype, stream) -> int:
    return lib().la_decode_step(q, k, v, out, state, zstate, B, H, dk, dv, _fm(feature_map),
                                normalize, level_weights, num_levels, t, dtype, stream)


def la_decode_state_elems(B, H, dk, dv, feature_map, num_levels):
    ze = ctypes.c_longlong()
    n = lib().la_decode_state_elems(B, H, dk, dv, _fm(feature_map), num_levels, ctypes.byref(ze))
    return n, ze.value


def la_noncausal_fwd(q, k, v, out, B, H, L, dk, dv, feature_map, normalize, dtype, workspace,
                     workspace_bytes, stream) -> int:
    return lib().la_noncausal_fwd(q, k, v, out, B, H, L, dk, dv, _fm(feature_map), normalize,
                                  dtype, workspace, workspace_bytes, stream)


def la_noncausal_workspace_bytes(B, H, L, dk, dv, feature_map, normalize, dtype) -> int:
    return lib().la_noncausal_workspace_bytes(B, H, L, dk, dv, _fm(feature_map), normalize, dtype)


def la_decay_fwd(q, k, v, out, B, H, L, dk, dv, C, feature_map, normalize, gamma, dtype,
                 workspace, workspace_bytes, stream, path) -> int:
    return lib().la_decay_fwd(q, k, v, out, B, H, L, dk, dv, C, _fm(feature_map), normalize,
                              gamma, dtype, workspace, workspace_bytes, stream, path)


def la_decay_decode_step(q, k, v, out, state, zstate, B, H, dk, dv, feature_map, normalize,
                         gamma, dtype, stream) -> int:
    return lib().la_decay_decode_step(q, k, v, out, state, zstate, B, H, dk, dv,
                                      _fm(feature_map), normalize, gamma, dtype, stream)


def la_decay_workspace_bytes(B, H, L, dk, dv, C, feature_map, normalize, gamma, dtype) -> int:
    return lib().la_decay_workspace_bytes(B, H, L, dk, dv, C, _fm(feature_map), normalize,
                                          gamma, dtype)


def la_decay_plan(B, H, L, dk, dv, C, feature_map, normalize, gamma, dtype, path, num_sms=0):
    info = la_plan_info()
    rc = lib().la_decay_plan(B, H, L, dk, dv, C, _fm(feature_map), normalize, gamma, dtype, path,
                             num_sms, ctypes.byref(info))
    return rc, info.as_dict()


def la_chunked_bwd(q, k, v, dout, dq, dk, dv, B, H, L, dk_, dv_, C, feature_map, normalize, gamma,
                   dtype, workspace, workspace_bytes, stream, path=LA_PATH_AUTO) -> int:
    return lib().la_chunked_bwd(q, k, v, dout, dq, dk, dv, B, H, L, dk_, dv_, C,
                                _fm(feature_map), normalize, gamma, dtype, workspace,
                                workspace_bytes, stream, path)


def la_chunked_bwd_ll(q, k, v, dout, dq, dk, dv, B, H, L, dk_, dv_, C, feature_map, normalize,
                      level_weights, num_levels, dtype, workspace, workspace_bytes, stream,
                      path=LA_PATH_AUTO) -> int:
    return lib().la_chunked_bwd_ll(q, k, v, dout, dq, dk, dv, B, H, L, dk_, dv_, C,
                                   _fm(feature_map), normalize, level_weights, num_levels, dtype,
                                   workspace, workspace_bytes, stream, path)


def la_chunked_bwd_ll_workspace_bytes(B, H, L, dk, dv, C, feature_map, normalize, num_levels,
                                      dtype) -> int:
    return lib().la_chunked_bwd_ll_workspace_bytes(B, H, L, dk, dv, C, _fm(feature_map),
                                                   normalize, num_levels, dtype)


def la_chunked_bwd_workspace_bytes(B, H, L, dk, dv, C, feature_map, normalize, dtype) -> int:
    return lib().la_chunked_bwd_workspace_bytes(B, H, L, dk, dv, C, _fm(feature_map), normalize,
                                                dtype)


def la_chunked_state(k, v, state, zstate, B, H, L, dk, dv, feature_map, gamma, dtype, stream) -> int:
    return lib().la_chunked_state(k, v, state, zstate, B, H, L, dk, dv, _fm(feature_map), gamma,
                                  dtype, stream)


def la_state_combine(state, zstate, seg_state, seg_zstate, B, H, D, dv, factor, stream) -> int:
    return lib().la_state_combine(state, zstate, seg_state, seg_zstate, B, H, D, dv, factor, stream)


def la_chunked_fwd_init(q, k, v, out, B, H, L, dk, dv, C, feature_map, normalize, gamma, state0,
                        zstate0, dtype, workspace, workspace_bytes, stream, path=LA_PATH_AUTO) -> int:
    return lib().la_chunked_fwd_init(q, k, v, out, B, H, L, dk, dv, C, _fm(feature_map), normalize,
                                     gamma, state0, zstate0, dtype, workspace, workspace_bytes,
                                     stream, path)


def la_version() -> str:
    return lib().la_version().decode()


# ---- torch-tensor convenience ----------------------------------------------------------
def noncausal_fwd(q, k, v, feature_map="identity", omega=None, normalize=False, out=None,
                  workspace=None, stream=None):
    """Bidirectional linear attention of CUDA tensors q,k [B,H,L,dk], v [B,H,L,dv]."""
    import torch
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    dtype = _dtype_code(q)
    if out is None:
        out = torch.empty((B, H, L, dv), dtype=q.dtype, device=q.device)
    fm = make_feature_map(feature_map, omega.shape[0] if omega is not None else 0,
                          omega.data_ptr() if omega is not None else 0)
    need = la_noncausal_workspace_bytes(B, H, L, dk, dv, fm, int(normalize), dtype)
    if need == 0:
        raise LAError(LA_ERR_UNSUPPORTED, "la_noncausal_workspace_bytes")
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = la_noncausal_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, L, dk,
                          dv, fm, int(normalize), dtype, workspace.data_ptr(), need, stream)
    if rc != LA_OK:
        raise LAError(rc, "la_noncausal_fwd")
    return out


def decode_state(B, H, dk, dv, feature_map="identity", m=0, num_levels=0, normalize=False,
                 device="cuda"):
    """Zero decoding state (and normaliser state when normalize) for la_decode_step."""
    import torch
    fm = make_feature_map(feature_map, m, 1 if feature_map == "favor" else 0)
    n, nz = la_decode_state_elems(B, H, dk, dv, fm, num_levels)
    if n == 0:
        raise LAError(LA_ERR_SHAPE, "la_decode_state_elems")
    S = torch.zeros(n, dtype=torch.float32, device=device)
    z = torch.zeros(nz, dtype=torch.float32, device=device) if normalize else None
    return S, z


def decode_step(q, k, v, state, zstate=None, t=0, feature_map="identity", omega=None,
                normalize=False, level_weights=None, out=None, stream=None):
    """One decoding step: q, k [B,H,dk], v [B,H,dv] CUDA tensors (one token per head);
    state / zstate from decode_state(); level_weights [B,H,NL] fp32 for the log-linear
    mask, with t the token position.  Returns out [B,H,dv]."""
    import torch
    B, H, dk = q.shape
    dv = v.shape[-1]
    dtype = _dtype_code(q)
    if out is None:
        out = torch.empty((B, H, dv), dtype=q.dtype, device=q.device)
    fm = make_feature_map(feature_map, omega.shape[0] if omega is not None else 0,
                          omega.data_ptr() if omega is not None else 0)
    nl = level_weights.shape[-1] if level_weights is not None else 0
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = la_decode_step(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                        state.data_ptr(), zstate.data_ptr() if zstate is not None else None,
                        B, H, dk, dv, fm, int(normalize),
                        level_weights.data_ptr() if level_weights is not None else None,
                        nl, int(t), dtype, stream)
    if rc != LA_OK:
        raise LAError(rc, "la_decode_step")
    return out



def decay_fwd(q, k, v, gamma, C=64, feature_map="identity", omega=None, normalize=False,
              out=None, workspace=None, stream=None, path=LA_PATH_AUTO):
    """Causal linear attention with the Retention decay gamma (la_decay_fwd) of CUDA
    tensors q,k [B,H,L,dk], v [B,H,L,dv]."""
    import torch
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA tensors")
    dtype = _dtype_code(q)
    if out is None:
        out = torch.empty((B, H, L, dv), dtype=q.dtype, device=q.device)
    fm = make_feature_map(feature_map, omega.shape[0] if omega is not None else 0,
                          omega.data_ptr() if omega is not None else 0)
    need = la_decay_workspace_bytes(B, H, L, dk, dv, C, fm, int(normalize), float(gamma), dtype)
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = la_decay_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, L, dk, dv,
                      C, fm, int(normalize), float(gamma), dtype,
                      workspace.data_ptr() if need else None, need, stream, path)
    if rc != LA_OK:
        raise LAError(rc, "la_decay_fwd")
    return out


def decay_decode_step(q, k, v, state, gamma, zstate=None, feature_map="identity", omega=None,
                      normalize=False, out=None, stream=None):
    """One decoding step with the Retention decay (la_decay_decode_step); state / zstate
    from decode_state().  Returns out [B,H,dv]."""
    import torch
    B, H, dk = q.shape
    dv = v.shape[-1]
    dtype = _dtype_code(q)
    if out is None:
        out = torch.empty((B, H, dv), dtype=q.dtype, device=q.device)
    fm = make_feature_map(feature_map, omega.shape[0] if omega is not None else 0,
                          omega.data_ptr() if omega is not None else 0)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = la_decay_decode_step(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              state.data_ptr(), zstate.data_ptr() if zstate is not None else None,
                              B, H, dk, dv, fm, int(normalize), float(gamma), dtype, stream)
    if rc != LA_OK:
        raise LAError(rc, "la_decay_decode_step")
    return out


def chunked_bwd(q, k, v, dout, C=64, feature_map="identity", omega=None, normalize=False,
                gamma=1.0, workspace=None, stream=None, path=LA_PATH_AUTO):
    """(dq, dk, dv) of the causal forward for CUDA tensors q,k [B,H,L,dk], v, dout [B,H,L,dv]."""
    import torch
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    dtype = _dtype_code(q)
    fm = make_feature_map(feature_map, omega.shape[0] if omega is not None else 0,
                          omega.data_ptr() if omega is not None else 0)
    need = la_chunked_bwd_workspace_bytes(B, H, L, dk, dv, C, fm, int(normalize), dtype)
    if need == 0:
        raise LAError(LA_ERR_UNSUPPORTED, "la_chunked_bwd_workspace_bytes")
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    dq, dk_t, dv_t = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = la_chunked_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(),
                        dq.data_ptr(), dk_t.data_ptr(), dv_t.data_ptr(), B, H, L, dk, dv, C, fm,
                        int(normalize), float(gamma), dtype, workspace.data_ptr(), need, stream,
                        path)
    if rc != LA_OK:
        raise LAError(rc, "la_chunked_bwd")
    return dq, dk_t, dv_t


def chunked_bwd_ll(q, k, v, dout, level_weights, C=64, feature_map="identity", omega=None,
                   normalize=False, workspace=None, stream=None, path=LA_PATH_AUTO):
    """(dq, dk, dv) of the log-linear forward (level_weights [B,H,L,NL] fp32 CUDA tensor)."""
    import torch
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    dtype = _dtype_code(q)
    nl = level_weights.shape[-1]
    fm = make_feature_map(feature_map, omega.shape[0] if omega is not None else 0,
                          omega.data_ptr() if omega is not None else 0)
    need = la_chunked_bwd_ll_workspace_bytes(B, H, L, dk, dv, C, fm, int(normalize), nl, dtype)
    if need == 0:
        raise LAError(LA_ERR_UNSUPPORTED, "la_chunked_bwd_ll_workspace_bytes")
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    dq, dk_t, dv_t = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = la_chunked_bwd_ll(q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(),
                           dq.data_ptr(), dk_t.data_ptr(), dv_t.data_ptr(), B, H, L, dk, dv, C, fm,
                           int(normalize), level_weights.data_ptr(), nl, dtype,
                           workspace.data_ptr(), need, stream, path)
    if rc != LA_OK:
        raise LAError(rc, "la_chunked_bwd_ll")
    return dq, dk_t, dv_t


def chunked_state(k, v, feature_map="identity", omega=None, gamma=1.0, normalize=True,
                  stream=None):
    """(state [B,H,D,dv], zstate [B,H,D] or None) a causal pass over k, v ends with."""
    import torch
    B, H, L, dk = k.shape
    dv = v.shape[-1]
    D = omega.shape[0] if omega is not None else dk
    S = torch.empty((B, H, D, dv), dtype=torch.float32, device=k.device)
    z = torch.empty((B, H, D), dtype=torch.float32, device=k.device) if normalize else None
    fm = make_feature_map(feature_map, D if omega is not None else 0,
                          omega.data_ptr() if omega is not None else 0)
    if stream is None:
        stream = torch.cuda.current_stream(k.device).cuda_stream
    rc = la_chunked_state(k.data_ptr(), v.data_ptr(), S.data_ptr(),
                          z.data_ptr() if z is not None else None, B, H, L, dk, dv, fm,
                          float(gamma), _dtype_code(k), stream)
    if rc != LA_OK:
        raise LAError(rc, "la_chunked_state")
    return S, z


def chunked_fwd_init(q, k, v, state0, zstate0=None, C=64, feature_map="identity", omega=None,
                     normalize=False, gamma=1.0, out=None, workspace=None, stream=None,
                     path=LA_PATH_AUTO):
    """The causal forward of q, k, v started from state0 [B,H,D,dv] (zstate0 [B,H,D])."""
    import torch
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    dtype = _dtype_code(q)
    if out is None:
        out = torch.empty((B, H, L, dv), dtype=q.dtype, device=q.device)
    fm = make_feature_map(feature_map, omega.shape[0] if omega is not None else 0,
                          omega.data_ptr() if omega is not None else 0)
    if gamma == 1.0:
        need = la_chunked_workspace_bytes(B, H, L, dk, dv, C, fm, int(normalize), 0, dtype)
    else:
        need = la_decay_workspace_bytes(B, H, L, dk, dv, C, fm, int(normalize), float(gamma), dtype)
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = la_chunked_fwd_init(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, L, dk,
                             dv, C, fm, int(normalize), float(gamma),
                             state0.data_ptr() if state0 is not None else None,
                             zstate0.data_ptr() if zstate0 is not None else None, dtype,
                             workspace.data_ptr() if need else None, need, stream, path)
    if rc != LA_OK:
        raise LAError(rc, "la_chunked_fwd_init")
    return out


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return LA_BF16
    if t.dtype == torch.float32:
        return LA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


_GENERIC_WARN_TOKENS = 1 << 20
_warned_shapes = set()


def _warn_if_generic(B, H, L, dk, dv, C, fm, normalize, nl, dtype, path):
    """The automatic path falls back to the generic CUDA-core kernel for shapes outside the
    tensor-core kernels' coverage; on large bf16 problems that is 100-1000x slower, so say so
    (once per shape) instead of staying silent."""
    if path != LA_PATH_AUTO or dtype != LA_BF16 or B * H * L < _GENERIC_WARN_TOKENS:
        return
    rc, info = la_chunked_plan(B, H, L, dk, dv, C, fm, normalize, int(nl > 0), nl, dtype,
                               LA_PATH_AUTO, 0)
    key = (B, H, L, dk, dv, C, fm.kind, fm.m, normalize, nl)
    if rc == LA_OK and info["path"] == LA_PATH_SIMT and key not in _warned_shapes:
        import warnings
        _warned_shapes.add(key)
        warnings.warn(f"la_chunked_fwd: B={B} H={H} L={L} dk={dk} dv={dv} C={C} runs on the generic "
                      "CUDA-core path (outside the tensor-core kernels' coverage, see "
                      "la_chunked_fwd_path in la_chunked.h); expect it to be 100-1000x slower",
                      RuntimeWarning, stacklevel=3)


def chunked_fwd(q, k, v, C=64, feature_map="identity", omega=None, normalize=False,
                level_weights=None, out=None, workspace=None, stream=None, path=LA_PATH_AUTO):
    """out[B,H,L,dv] = chunkwise causal linear attention of CUDA tensors q,k [B,H,L,dk],
    v [B,H,L,dv] (bf16 or fp32, contiguous).  omega: [m, dk] fp32 CUDA tensor for
    feature_map="favor".  level_weights: [B,H,L,NL] fp32 CUDA tensor for the log-linear
    mask.  out / workspace are allocated with torch when not given."""
    import torch
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA tensors")
    dtype = _dtype_code(q)
    if out is None:
        out = torch.empty((B, H, L, dv), dtype=q.dtype, device=q.device)
    fm = make_feature_map(feature_map, omega.shape[0] if omega is not None else 0,
                          omega.data_ptr() if omega is not None else 0)
    nl = level_weights.shape[-1] if level_weights is not None else 0
    _warn_if_generic(B, H, L, dk, dv, C, fm, int(normalize), nl, dtype, path)
    need = la_chunked_workspace_bytes(B, H, L, dk, dv, C, fm, int(normalize), nl, dtype)
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = la_chunked_fwd_path(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, L,
                             dk, dv, C, fm, int(normalize),
                             level_weights.data_ptr() if level_weights is not None else None,
                             nl, dtype, workspace.data_ptr() if need else None,
                             need, stream, path)
    if rc != LA_OK:
        raise LAError(rc, "la_chunked_fwd")
    return out
