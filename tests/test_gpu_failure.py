"""Failure detection on the GPU without a GPU fault.

A test-only knob makes the feature-map warps of the tensor-core kernel never signal, so
the MMA warp's bounded wait runs out.  The kernel must record LA_ERR_TIMEOUT in the device
error word, drain its own copies and MMAs, release TMEM and return; the context must stay
usable (a normal call right after gives the right answer).
"""
import os

import numpy as np
import pytest

import synth
from parity_util import assert_close, oracle_heads, run_gpu, workload

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


def test_stalled_wait_times_out_and_context_survives(la_mod):
    import time

    import torch
    la = la_mod
    w = workload("elu1-norm-d128-L8192", B=1, H=2, L=512)
    inp = synth.make_inputs(w, seed=9)
    B, H, L, d = w["B"], w["H"], w["L"], w["dk"]
    q = torch.from_numpy(inp["q"].view(np.int16)).view(torch.bfloat16).reshape(B, H, L, d).cuda()
    k = torch.from_numpy(inp["k"].view(np.int16)).view(torch.bfloat16).reshape(B, H, L, d).cuda()
    v = torch.from_numpy(inp["v"].view(np.int16)).view(torch.bfloat16).reshape(B, H, L, d).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    assert la.la_last_device_status(stream) == la.LA_OK
    os.environ["LA_DEBUG_STALL"] = "1"
    os.environ["LA_DEBUG_TIMEOUT_NS"] = "200000000"  # 0.2 s
    try:
        t0 = time.time()
        la.chunked_fwd(q, k, v, C=64, feature_map="elu1", normalize=True, path=la.LA_PATH_TC)
        st = la.la_last_device_status(stream)
        elapsed = time.time() - t0
    finally:
        del os.environ["LA_DEBUG_STALL"]
        del os.environ["LA_DEBUG_TIMEOUT_NS"]
    assert st == la.LA_ERR_TIMEOUT, la.la_status_string(st)
    assert elapsed < 30
    # the error word was cleared by the read, and the context still works
    assert la.la_last_device_status(stream) == la.LA_OK
    out, _ = run_gpu(w, inp, 64, la.LA_PATH_TC)
    assert_close(out, oracle_heads(w, inp, [0, 1]), "after timeout")
