"""Each stage alone through its own C-ABI entry point, against the oracle.

* ssd_chunk_cumsum vs the float64 within-chunk cumsum (section "Kernel 1");
  dt_t must be dt transposed exactly.
* ssd_state_pass vs the oracle's chunk start states and final state
  (section "Kernel 2: fwd_pass_state").
* ssd_chunk_out fed the ORACLE's chunk states, vs the oracle's y
  (section "Kernel 3: compute_out"), so a stage-3 error cannot hide behind
  a stage-2 one.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL, assert_parity, case_inputs, oracle_run, to_gpu
import state_space_sequence_cumsum_gb300 as ssd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("L,H,T", [(1, 1, 64), (300, 3, 64), (1000, 80, 256), (4095, 33, 128),
                                   (77, 5, 16)])
def test_chunk_cumsum(L, H, T):
    inp = case_inputs(2, L, H, 4, 4, 1, T, seed=L)
    g = to_gpu(inp)
    G, dtT = ssd.ssd_chunk_cumsum(g["dt"], g["A"], T)
    ref = oracle.chunk_cumsum(inp["dt"], inp["A"], T)
    err = np.max(np.abs(G.cpu().double().numpy() - ref))
    assert err <= 1e-5 * max(1.0, np.max(np.abs(ref))), err
    assert torch.equal(dtT.cpu(), inp["dt"].permute(0, 2, 1).contiguous())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,L,H,P,S,G,T", [(2, 520, 4, 64, 128, 1, 128),
                                           (1, 700, 6, 32, 64, 3, 256),
                                           (1, 257, 2, 16, 16, 1, 64),
                                           (1, 300, 2, 128, 192, 1, 256),   # ragged dstate slice
                                           (2, 1000, 4, 64, 64, 2, 256),    # half-empty slice
                                           (1, 129, 3, 64, 256, 3, 128),    # tile + 1 token
                                           (1, 4095, 2, 64, 128, 1, 256),   # ragged, many tiles
                                           (1, 2900, 2, 64, 128, 1, 128),   # segments, short last
                                           (1, 6000, 1, 128, 256, 1, 256)])  # segments, two tiles a chunk
def test_state_pass(dtype, B, L, H, P, S, G, T):
    inp = case_inputs(B, L, H, P, S, G, T, dtype=dtype, init="randn", seed=L + P)
    g = to_gpu(inp)
    Gc, dtT = ssd.ssd_chunk_cumsum(g["dt"], g["A"], T)
    st, fin = ssd.ssd_state_pass(g["x"], g["B"], dtT, Gc, T, init_state=g["init"])
    ref = oracle_run(inp, T, want_states=True)
    assert_parity(st, ref["chunk_states"], dtype, "chunk_states")
    assert_parity(fin, ref["final_state"], dtype, "final_state")
    assert torch.equal(st[:, :, 0].cpu(), inp["init"])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,L,H,P,S,G,T", [(2, 520, 4, 64, 128, 1, 128),
                                           (1, 700, 6, 32, 64, 3, 256),
                                           (1, 100, 2, 128, 256, 2, 64),
                                           (1, 600, 4, 64, 128, 2, 256),   # two tiles per chunk
                                           (2, 333, 2, 128, 128, 1, 256),
                                           (1, 260, 4, 64, 256, 1, 128),
                                           (1, 390, 2, 64, 64, 2, 256),
                                           (1, 200, 2, 128, 64, 1, 128),
                                           (2, 645, 4, 64, 512, 2, 128),   # dstate blocks, ragged
                                           (1, 384, 3, 64, 384, 1, 128)])
def test_chunk_out_from_oracle_states(dtype, B, L, H, P, S, G, T):
    inp = case_inputs(B, L, H, P, S, G, T, dtype=dtype, init="randn", seed=L + S)
    g = to_gpu(inp)
    ref = oracle_run(inp, T, want_states=True)
    Gc, dtT = ssd.ssd_chunk_cumsum(g["dt"], g["A"], T)
    states = torch.from_numpy(ref["chunk_states"]).float().cuda()
    y = ssd.ssd_chunk_out(g["x"], g["B"], g["C"], dtT, Gc, states, g["D"], T)
    assert_parity(y, ref["y"], dtype, "y")


@pytest.mark.parametrize("init", ["zero", "randn"])
@pytest.mark.parametrize("B,L,H,P,S,G,T", [(1, 5000, 2, 64, 128, 1, 128),
                                           (1, 9000, 1, 64, 512, 1, 256),
                                           (2, 3333, 3, 128, 128, 3, 128)])
def test_segmented_and_plain_state_pass_agree(B, L, H, P, S, G, T, init, monkeypatch):
    """Few (batch, head) units and a long sequence split the tensor-core state
    pass into parallel segments; SSD_STATE_PASS=plain runs it unsplit.  Both
    follow "Kernel 2: fwd_pass_state", so they agree to f32 rounding and each
    matches the oracle."""
    inp = case_inputs(B, L, H, P, S, G, T, init=init, seed=L + S + P)
    g = to_gpu(inp)
    Gc, dtT = ssd.ssd_chunk_cumsum(g["dt"], g["A"], T)
    init_state = g["init"] if init == "randn" else None
    st, fin = ssd.ssd_state_pass(g["x"], g["B"], dtT, Gc, T, init_state=init_state)
    monkeypatch.setenv("SSD_STATE_PASS", "plain")
    st_p, fin_p = ssd.ssd_state_pass(g["x"], g["B"], dtT, Gc, T, init_state=init_state)
    assert ssd.ssd_stream_status() == 0
    scale = max(1.0, fin_p.abs().max().item())
    assert (st - st_p).abs().max().item() <= 1e-4 * scale
    assert (fin - fin_p).abs().max().item() <= 1e-4 * scale
    ref = oracle_run(inp, T, want_states=True)
    assert_parity(st, ref["chunk_states"], torch.bfloat16, "chunk_states")
    assert_parity(fin, ref["final_state"], torch.bfloat16, "final_state")


def test_state_pass_without_outputs_is_a_noop():
    inp = case_inputs(1, 128, 2, 64, 64, 1, 64, seed=3)
    g = to_gpu(inp)
    Gc, dtT = ssd.ssd_chunk_cumsum(g["dt"], g["A"], 64)
    st, fin = ssd.ssd_state_pass(g["x"], g["B"], dtT, Gc, 64, chunk_states=None,
                                 final_state=None)
    assert st is None and fin is None
    assert ssd.ssd_stream_status() == 0


@pytest.mark.parametrize("B,L,H,P,S,G,T", [(2, 700, 4, 64, 128, 2, 256),
                                           (1, 513, 2, 64, 64, 1, 128),
                                           (1, 300, 4, 64, 256, 4, 128),
                                           (3, 2000, 5, 64, 128, 1, 256)])  # several segments
def test_fused_state_out_with_chunk_states(B, L, H, P, S, G, T):
    """Fused stages 2+3 through ssd_state_out: y, final and every chunk state."""
    inp = case_inputs(B, L, H, P, S, G, T, init="randn", seed=L + S)
    g = to_gpu(inp)
    Gc, dtT = ssd.ssd_chunk_cumsum(g["dt"], g["A"], T)
    y, fin, st = ssd.ssd_state_out(g["x"], g["B"], g["C"], dtT, Gc, g["D"], T,
                                   initial_state=g["init"], chunk_states=True)
    assert ssd.ssd_stream_status() == 0
    ref = oracle_run(inp, T, want_states=True)
    assert_parity(y, ref["y"], torch.bfloat16, "y")
    assert_parity(fin, ref["final_state"], torch.bfloat16, "final_state")
    assert_parity(st, ref["chunk_states"], torch.bfloat16, "chunk_states")


def test_state_out_rejects_f32():
    inp = case_inputs(1, 64, 2, 64, 64, 1, 128, dtype=torch.float32)
    g = to_gpu(inp)
    Gc, dtT = ssd.ssd_chunk_cumsum(g["dt"], g["A"], 128)
    with pytest.raises(ssd.SsdError):
        ssd.ssd_state_out(g["x"], g["B"], g["C"], dtT, Gc, g["D"], 128)
