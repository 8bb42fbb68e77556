"""GPU parity of the single-token decode step (ssd_decode_step) against the
float64 oracle.

The decode step is the recurrence of section "Mamba-2 架构" taken one token
at a time on a carried state.  Each case runs several steps on the GPU,
feeding every step's state into the next, and compares every step's y and
the last state with the oracle run over the same tokens from the same
initial state.  The state update is f32 arithmetic on exactly widened
inputs, so the state is held to 1e-5 * rms even for bf16 inputs; y is held
to the usual per-dtype tolerance (it is rounded to the input dtype).
"""
import pytest
import torch

import oracle
from parity_util import TOL, rel_err
import state_space_sequence_cumsum_gb300 as ssd
from state_space_sequence_cumsum_gb300.inputs import Shape, make_inputs

pytestmark = pytest.mark.gpu

STATE_TOL = 1e-5


def step_inputs(g, t):
    return (g["x"][:, t:t + 1].contiguous(), g["dt"][:, t:t + 1].contiguous(),
            g["B"][:, t:t + 1].contiguous(), g["C"][:, t:t + 1].contiguous())


def run_steps(B, H, P, S, G, steps, dtype, in_place=True, seed=0):
    inp = make_inputs(Shape(B, steps, H, P, S, G, 64), dtype=dtype, init="randn", seed=seed,
                      init_std=0.5)
    g = {k: v.cuda() for k, v in inp.items()}
    state = g["init"].clone()
    ys = []
    for t in range(steps):
        x, dt, Bt, Ct = step_inputs(g, t)
        out = None if in_place else torch.empty_like(state)
        y, new_state = ssd.ssd_decode_step(x, dt, g["A"], Bt, Ct, g["D"], state, state_out=out)
        assert (new_state.data_ptr() == state.data_ptr()) == in_place
        state = new_state
        ys.append(y)
    torch.cuda.synchronize()
    assert ssd.ssd_stream_status() == 0
    ref = oracle.fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], 64,
                     init=inp["init"])
    return torch.cat(ys, dim=1), state, ref


@pytest.mark.parametrize("B,H,P,S,G,steps,dtype", [
    (4, 80, 64, 128, 1, 3, torch.bfloat16),   # one token of the 2.7B-layer shape
    (2, 8, 64, 128, 4, 4, torch.float32),
    (3, 6, 32, 64, 3, 2, torch.bfloat16),     # grouped B / C
    (1, 4, 16, 512, 1, 2, torch.bfloat16),    # largest dstate: four vectors per lane
    (2, 4, 16, 256, 2, 2, torch.float32),
    (1, 2, 16, 16, 1, 5, torch.float32),      # four lanes per row
    (2, 4, 16, 80, 1, 2, torch.float32),      # five vectors per lane: one warp per row
    (2, 3, 8, 17, 1, 3, torch.bfloat16),      # dstate not a multiple of 4
])
def test_decode_steps_match_oracle(B, H, P, S, G, steps, dtype):
    y, state, ref = run_steps(B, H, P, S, G, steps, dtype)
    assert rel_err(y, ref["y"]) <= TOL[dtype]
    assert rel_err(state, ref["final_state"]) <= STATE_TOL


def test_decode_separate_state_buffer():
    y, state, ref = run_steps(2, 8, 64, 128, 1, 3, torch.bfloat16, in_place=False, seed=3)
    assert rel_err(y, ref["y"]) <= TOL[torch.bfloat16]
    assert rel_err(state, ref["final_state"]) <= STATE_TOL


def test_decode_zero_dt_keeps_state():
    """dt = 0: no decay and no input, so the state is unchanged bit for bit and
    y = C h + D x."""
    inp = make_inputs(Shape(2, 1, 4, 32, 64, 2, 64), dtype=torch.float32, init="randn", seed=5)
    g = {k: v.cuda() for k, v in inp.items()}
    dt0 = torch.zeros_like(g["dt"])
    state = g["init"].clone()
    y, _ = ssd.ssd_decode_step(g["x"], dt0, g["A"], g["B"], g["C"], g["D"], state)
    torch.cuda.synchronize()
    assert torch.equal(state, g["init"])
    ref = oracle.fwd(inp["x"], dt0.cpu(), inp["A"], inp["B"], inp["C"], inp["D"], 64,
                     init=inp["init"])
    assert rel_err(y, ref["y"]) <= TOL[torch.float32]


def test_decode_continues_a_forward_pass():
    """Generation: ssd_fwd over a 1000-token prompt, then three decode steps
    from its final state, against the oracle over all 1003 tokens."""
    L0, steps = 1000, 3
    shape = Shape(2, L0 + steps, 16, 64, 128, 1, 128)
    inp = make_inputs(shape, dtype=torch.bfloat16, seed=9)
    g = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    pre = {k: g[k][:, :L0].contiguous() for k in ("x", "dt", "B", "C")}
    _, state, _ = ssd.ssd_fwd(pre["x"], pre["dt"], g["A"], pre["B"], pre["C"], g["D"],
                              chunk_size=128, return_final_state=True)
    ys = []
    for t in range(L0, L0 + steps):
        x, dt, Bt, Ct = step_inputs(g, t)
        y, state = ssd.ssd_decode_step(x, dt, g["A"], Bt, Ct, g["D"], state)
        ys.append(y)
    torch.cuda.synchronize()
    assert ssd.ssd_stream_status() == 0
    ref = oracle.fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], 128)
    tol = TOL[torch.bfloat16]
    assert rel_err(torch.cat(ys, dim=1), ref["y"][:, L0:]) <= tol
    assert rel_err(state, ref["final_state"]) <= tol


def test_decode_token_slices_of_a_sequence():
    """Per-token views of [1, L, ...] tensors, no copies: dt's view starts at
    a 4-byte boundary only, which this entry point accepts."""
    inp = make_inputs(Shape(1, 3, 3, 16, 32, 1, 64), dtype=torch.float32, init="randn", seed=11,
                      init_std=0.5)
    g = {k: v.cuda() for k, v in inp.items()}
    state = g["init"].clone()
    ys = []
    for t in range(3):
        y, state = ssd.ssd_decode_step(g["x"][:, t:t + 1], g["dt"][:, t:t + 1], g["A"],
                                       g["B"][:, t:t + 1], g["C"][:, t:t + 1], g["D"], state)
        ys.append(y)
    torch.cuda.synchronize()
    ref = oracle.fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], 64,
                     init=inp["init"])
    assert rel_err(torch.cat(ys, dim=1), ref["y"]) <= TOL[torch.float32]
    assert rel_err(state, ref["final_state"]) <= STATE_TOL
