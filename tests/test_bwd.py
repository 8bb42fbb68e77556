"""GPU parity of the backward pass (ssd_bwd) against the oracle's adjoint.

The oracle (``oracle.bwd``) computes every gradient in float64 by the
adjoint of the token recurrence, pinned by finite differences
(test_oracle_bwd.py).  The GPU computes in f32 from the same (exactly
widened) inputs, so every gradient is held to 1e-4 * rms (the f32 bound of
the forward's parity tests) -- except that outputs in a bf16 call's dtype
(dx, dB, dC) are then rounded to bf16.  dB and dC have heavy-tailed
magnitudes (max / rms of 10-17 on these inputs), so that rounding alone
moves them by up to ~6e-2 * rms: those outputs are held element by element
to the rounding bound, |gpu - oracle| <= 2^-8 |oracle| + 1e-4 * rms.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import rel_err
import state_space_sequence_cumsum_gb300 as ssd
from state_space_sequence_cumsum_gb300.inputs import Shape, make_inputs

pytestmark = pytest.mark.gpu

F32_TOL = 1e-4


def run_case(B, L, H, P, S, G, dtype, init=True, dfinal=True, seed=0):
    inp = make_inputs(Shape(B, L, H, P, S, G, 64), dtype=dtype, init="randn" if init else "zero",
                      seed=seed, init_std=0.5)
    rng = np.random.default_rng(seed + 7)
    dy = torch.from_numpy(rng.standard_normal((B, L, H, P)).astype(np.float32)).to(dtype)
    df = (torch.from_numpy(rng.standard_normal((B, H, P, S)).astype(np.float32))
          if dfinal else None)
    g = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    out = ssd.ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], dy.cuda(),
                      initial_state=g["init"], dfinal=None if df is None else df.cuda())
    torch.cuda.synchronize()
    assert ssd.ssd_stream_status() == 0
    ref = oracle.bwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], dy,
                     init=inp["init"], dfinal=df)
    return out, ref


def check(out, ref, dtype):
    for k in ("dx", "dB", "dC"):
        if dtype == torch.float32:
            e = rel_err(out[k], ref[k])
            assert e <= F32_TOL, f"{k}: max|err|/rms = {e:.3e}"
        else:  # the f32 result rounded to bf16
            g = out[k].detach().to("cpu", torch.float64).numpy()
            r = ref[k]
            rms = float(np.sqrt(np.mean(r * r)))
            excess = np.abs(g - r) - (2.0 ** -8 * np.abs(r) + F32_TOL * rms)
            assert np.max(excess) <= 0.0, f"{k}: beyond the bf16 rounding bound by {np.max(excess):.3e}"
    for k in ("ddt", "dA", "dD", "dinit"):
        e = rel_err(out[k], ref[k])
        assert e <= F32_TOL, f"{k}: max|err|/rms = {e:.3e}"


@pytest.mark.parametrize("B,L,H,P,S,G,dtype", [
    (2, 200, 4, 16, 32, 2, torch.float32),     # ragged last chunk, grouped B / C
    (2, 200, 4, 16, 32, 2, torch.bfloat16),
    (1, 64, 2, 64, 128, 1, torch.bfloat16),    # one whole chunk
    (2, 300, 8, 64, 128, 2, torch.bfloat16),   # 2.7B-layer head shape
    (1, 130, 2, 64, 256, 1, torch.float32),    # four dstate tiles
    (1, 70, 2, 32, 512, 1, torch.bfloat16),    # largest dstate
    (3, 1, 3, 8, 16, 3, torch.float32),        # one token
])
def test_bwd_matches_oracle(B, L, H, P, S, G, dtype):
    out, ref = run_case(B, L, H, P, S, G, dtype)
    check(out, ref, dtype)


def test_bwd_without_initial_state_or_final_gradient():
    out, ref = run_case(2, 150, 4, 32, 64, 1, torch.float32, init=False, dfinal=False, seed=4)
    check(out, ref, torch.float32)


def test_autograd_function():
    """torch.autograd through SsdFunction (ssd_fwd forward, ssd_bwd backward)."""
    B, L, H, P, S, G = 2, 257, 4, 64, 128, 1
    inp = make_inputs(Shape(B, L, H, P, S, G, 64), dtype=torch.bfloat16, init="randn", seed=12,
                      init_std=0.5)
    rng = np.random.default_rng(3)
    wy = torch.from_numpy(rng.standard_normal((B, L, H, P)).astype(np.float32))
    wf = torch.from_numpy(rng.standard_normal((B, H, P, S)).astype(np.float32))
    g = {k: v.cuda().requires_grad_(True) for k, v in inp.items()}
    y, final = ssd.SsdFunction.apply(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["init"])
    loss = (y.float() * wy.cuda()).sum() + (final * wf.cuda()).sum()
    loss.backward()
    torch.cuda.synchronize()
    ref = oracle.bwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                     wy.to(torch.bfloat16), init=inp["init"], dfinal=wf)
    got = {"dx": g["x"].grad, "ddt": g["dt"].grad, "dA": g["A"].grad, "dB": g["B"].grad,
           "dC": g["C"].grad, "dD": g["D"].grad, "dinit": g["init"].grad}
    check(got, ref, torch.bfloat16)
