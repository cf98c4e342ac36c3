"""The no-allocation entry point, checked against the main entry point on the GPU.

Some callers cannot allocate device memory (code inside an allocator or memory-pool
callback, plugins whose host application owns every allocation, real-time loops that must
not call cudaMalloc).  la_chunked_fwd_noalloc serves them from a fixed scratch buffer in the
library: every plan that needs scratch uses it (sequences cut into segments on the tensor-core
paths, the log-linear mask's level states).  This file is collected last so that, if it fails, a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest

import synth
from parity_util import MAX_ABS_FRAC, REL_RMS, from_device, to_device, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def la_mod():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunkwise_causal_linear_gb300 import build
    build.build()
    import chunkwise_causal_linear_gb300 as la
    return la


# Problems whose plan needs scratch: the log-linear mask (three heads: level states and a
# sequence cut into segments), and elu+1 with the normaliser on one d = 128 head, where the
# tensor-core path cuts the sequence into segments and keeps their fp32 totals in scratch.
NOALLOC_CASES = [
    ("loglinear-d64-L65536", dict(B=1, H=3, L=1500)),
    ("elu1-norm-d128-L8192", dict(B=1, H=1, L=8192)),
]


@pytest.mark.parametrize("name,over", NOALLOC_CASES)
def test_noalloc_matches_main_entry_point_twice(la_mod, name, over):
    import torch
    la = la_mod
    w = workload(name, **over)
    B, H, L, dk, dv = w["B"], w["H"], w["L"], w["dk"], w["dv"]
    C = 64
    fm = la.make_feature_map(w["fm"])
    norm = int(w["normalize"])
    stream = torch.cuda.current_stream().cuda_stream
    for call, seed in enumerate((21, 22)):  # two calls in a row on the shared scratch
        inp = synth.make_inputs(w, seed=seed)
        q = to_device(inp["q"], "bf16", (B, H, L, dk))
        k = to_device(inp["k"], "bf16", (B, H, L, dk))
        v = to_device(inp["v"], "bf16", (B, H, L, dv))
        lam = None if inp["lam"] is None else torch.from_numpy(inp["lam"]).reshape(B, H, L, -1).cuda()
        nl = 0 if lam is None else lam.shape[-1]
        lp = None if lam is None else lam.data_ptr()
        need = la.la_chunked_workspace_bytes(B, H, L, dk, dv, C, fm, norm, nl, la.LA_BF16)
        assert need > 0
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        ref = torch.empty_like(v)
        got = torch.full_like(v, float("nan"))
        rc = la.la_chunked_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), ref.data_ptr(), B, H, L,
                               dk, dv, C, fm, norm, lp, nl, la.LA_BF16, ws.data_ptr(), need, stream)
        assert rc == la.LA_OK, la.la_status_string(rc)
        rc = la.la_chunked_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), got.data_ptr(),
                                       B, H, L, dk, dv, C, fm, norm, lp, nl, la.LA_BF16, stream)
        assert rc == la.LA_OK, la.la_status_string(rc)
        torch.cuda.synchronize()
        assert la.la_last_device_status(stream) == la.LA_OK
        a, b = from_device(got), from_device(ref)
        assert np.isfinite(a).all(), f"call {call}"
        err = np.abs(a - b)
        assert err.max() <= MAX_ABS_FRAC * np.abs(b).max(), f"call {call}"
        assert np.linalg.norm(a - b) <= REL_RMS * np.linalg.norm(b), f"call {call}"


def test_noalloc_rejects_problems_beyond_its_scratch(la_mod):
    import torch
    la = la_mod
    fm = la.make_feature_map("identity")
    # 256 heads of L = 65,536, d = 64: about 44 MB of level states, beyond the 8 MiB buffer
    B, H, L, d = 16, 16, 65536, 64
    need = la.la_chunked_workspace_bytes(B, H, L, d, d, 64, fm, 0, 17, la.LA_BF16)
    assert need > 8 << 20
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")  # never read: rejected first
    p = dummy.data_ptr()
    rc = la.la_chunked_fwd_noalloc(p, p, p, p, B, H, L, d, d, 64, fm, 0, p, 17, la.LA_BF16,
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == la.LA_ERR_SCRATCH_LIMIT
    assert "8 MiB" in la.la_status_string(rc)
