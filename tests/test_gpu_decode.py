"""The recurrent decoding step (la_decode_step) against the oracle.

Stepping t = 0..L-1 through la_decode_step is the recurrent form of the same function the
chunked forward computes ("Linear Attention / Performerの理論と実装", "再帰的な状態更新";
"論文紹介：Log Linear Attention", slides 17-22), so every step's output is compared with the
oracle's output row t for the whole sequence.
"""
import numpy as np
import pytest

import synth
from parity_util import assert_close, oracle_heads, to_device, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunkwise_causal_linear_gb300 import build
    build.build()


def decode_all(w, inp):
    """Runs la_decode_step for every position; returns [B*H, L, dv] float64."""
    import torch

    import chunkwise_causal_linear_gb300 as la
    B, H, L, dk, dv = w["B"], w["H"], w["L"], w["dk"], w["dv"]
    q = to_device(inp["q"], w["dtype"], (B, H, L, dk))
    k = to_device(inp["k"], w["dtype"], (B, H, L, dk))
    v = to_device(inp["v"], w["dtype"], (B, H, L, dv))
    omega = None if inp["omega"] is None else torch.from_numpy(inp["omega"]).cuda()
    lam = None
    if inp["lam"] is not None:
        lam_np = inp["lam"].reshape(B, H, L, -1)
        # the step after token L-1 builds the state for position L: give the levels room for
        # it with zero-weight levels (they hold nothing any earlier row reads)
        r_last = (L & -L).bit_length() - 1
        if r_last + 2 > lam_np.shape[-1]:
            pad = np.zeros(lam_np.shape[:-1] + (r_last + 2 - lam_np.shape[-1],), dtype=lam_np.dtype)
            lam_np = np.concatenate([lam_np, pad], axis=-1)
        lam = torch.from_numpy(np.ascontiguousarray(lam_np)).cuda()
    nl = lam.shape[-1] if lam is not None else 0
    S, z = la.decode_state(B, H, dk, dv, w["fm"], w["m"], nl, w["normalize"])
    outs = []
    for t in range(L):
        o = la.decode_step(q[:, :, t].contiguous(), k[:, :, t].contiguous(), v[:, :, t].contiguous(),
                           S, z, t=t, feature_map=w["fm"], omega=omega, normalize=w["normalize"],
                           level_weights=lam[:, :, t].contiguous() if lam is not None else None)
        outs.append(o.float())
    torch.cuda.synchronize()
    st = la.la_last_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == la.LA_OK, la.la_status_string(st)
    out = torch.stack(outs, dim=2)  # [B, H, L, dv]
    return out.reshape(B * H, L, dv).double().cpu().numpy()


CASES = [
    ("elu1-norm-d128-L8192", dict(B=1, H=2, L=70, dk=64, dv=48)),
    ("elu1-norm-d128-L8192", dict(B=2, H=1, L=40, normalize=False, dk=32, dv=72)),
    ("identity-d64-L2048", dict(B=1, H=3, L=50)),
    ("favor-m256-d64-L16384", dict(B=1, H=2, L=40)),
    ("favor-m256-d64-L16384", dict(B=1, H=1, L=30, normalize=False)),
    ("loglinear-d64-L65536", dict(B=1, H=2, L=100)),
    ("loglinear-d64-L65536", dict(B=1, H=1, L=64, dv=40)),
    # the benchmark's decoding configuration: all 128 heads of B8 H16 d128 per step
    ("elu1-norm-d128-L8192", dict(L=48)),
]


@pytest.mark.parametrize("base,over", CASES)
def test_decode_steps_match_oracle(base, over):
    w = workload(base, **over)
    inp = synth.make_inputs(w, seed=5)
    out = decode_all(w, inp)
    ref = oracle_heads(w, inp, list(range(w["B"] * w["H"])))
    assert_close(out, ref, f"decode {base} {over}")


def test_integer_decode_is_exact():
    """fp32 small-integer inputs: the recurrence's sums stay exact in fp32."""
    w = workload("tiny-int-exact", B=1, H=2, L=40, dk=8, dv=8)
    inp = synth.make_inputs(w, seed=6)
    out = decode_all(w, inp)
    ref = oracle_heads(w, inp, [0, 1], method="scores_first")
    assert np.array_equal(out, ref), np.abs(out - ref).max()


def test_decode_agrees_with_chunked_forward():
    """The two forms of one function: decode steps vs the chunked tensor-core forward."""
    from parity_util import run_gpu
    w = workload("elu1-norm-d128-L8192", B=1, H=2, L=200)
    inp = synth.make_inputs(w, seed=7)
    dec = decode_all(w, inp)
    fwd, _ = run_gpu(w, inp, 64, 0)
    assert_close(dec, fwd, "decode vs chunked")


def test_decode_refuses_levels_too_few_for_the_next_position():
    """Position t+1 = 64 needs level 7: with 7 levels the step reports LA_ERR_SHAPE and
    leaves the state untouched (nothing is launched)."""
    import torch

    import chunkwise_causal_linear_gb300 as la
    q = torch.zeros((1, 1, 8), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((1, 1, 8), dtype=torch.bfloat16, device="cuda")
    S, _ = la.decode_state(1, 1, 8, 8, num_levels=7)
    S.fill_(1.0)
    lam = torch.ones((1, 1, 7), dtype=torch.float32, device="cuda")
    with pytest.raises(la.LAError) as e:
        la.decode_step(q, q, v, S, t=63, level_weights=lam)
    assert e.value.status == la.LA_ERR_SHAPE
    la.decode_step(q, q, v, S, t=62, level_weights=lam)  # position 63 fits
    torch.cuda.synchronize()
