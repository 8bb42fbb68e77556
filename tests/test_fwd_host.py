"""ssd_fwd_host: the forward from host buffers to host buffers, its copies
overlapped with the kernels by cutting the sequence into parts of whole
chunks that carry the state ("Kernel 2: fwd_pass_state": the state passes
from chunk to chunk, so a cut at a chunk boundary with the carried state is
the same function).  Checked against the oracle and against ssd_fwd on the
device, over sequences cut into one, two and four parts (ragged last part)."""
import numpy as np
import pytest
import torch

from parity_util import assert_parity, case_inputs, oracle_run, to_gpu
import state_space_sequence_cumsum_gb300 as ssd

pytestmark = pytest.mark.gpu


def _pinned(inp):
    return {k: (None if v is None else v.contiguous().pin_memory()) for k, v in inp.items()}


@pytest.mark.parametrize("B,L,H,P,S,G,T,init", [(2, 300, 4, 64, 128, 1, 128, "randn"),    # one part
                                                 (1, 1100, 4, 64, 128, 2, 128, "zero"),    # two parts
                                                 (2, 4000, 6, 64, 64, 3, 256, "randn"),    # four, ragged
                                                 (3, 2100, 2, 32, 64, 1, 64, "randn")])    # f32 below
def test_fwd_host_matches_oracle_and_device(B, L, H, P, S, G, T, init):
    dtype = torch.float32 if P == 32 else torch.bfloat16
    inp = case_inputs(B, L, H, P, S, G, T, dtype=dtype, init=init, seed=L + H)
    hi = _pinned(inp)
    y, fin = ssd.ssd_fwd_host(hi["x"], hi["dt"], hi["A"], hi["B"], hi["C"], hi["D"],
                              chunk_size=T, initial_state=hi["init"])
    torch.cuda.synchronize()
    assert ssd.ssd_stream_status() == 0
    ref = oracle_run(inp, T)
    assert_parity(y, ref["y"], dtype, "y")
    assert_parity(fin, ref["final_state"], dtype, "final_state")
    g = to_gpu(inp)
    yd, fd, _ = ssd.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=T,
                            initial_state=g["init"])
    # the parts differ from the single call only in how the carried state is rounded
    scale = float(fd.abs().max())
    assert float((fin - fd.cpu()).abs().max()) <= 2e-3 * max(1.0, scale)


def test_fwd_host_repeat_calls_reuse_workspace():
    inp = case_inputs(2, 2048, 4, 64, 128, 1, 128, init="randn", seed=9)
    hi = _pinned(inp)
    ws = ssd.Workspace()
    outs = []
    for _ in range(3):
        y, fin = ssd.ssd_fwd_host(hi["x"], hi["dt"], hi["A"], hi["B"], hi["C"], hi["D"],
                                  chunk_size=128, initial_state=hi["init"], workspace=ws)
        torch.cuda.synchronize()
        outs.append((y.clone(), fin.clone()))
    assert ssd.ssd_stream_status() == 0
    for y, fin in outs[1:]:
        assert torch.equal(y, outs[0][0]) and torch.equal(fin, outs[0][1])


def test_fwd_host_empty_sequence_returns_init():
    inp = case_inputs(1, 0, 2, 64, 64, 1, 128, init="randn", seed=2)
    hi = _pinned(inp)
    y, fin = ssd.ssd_fwd_host(hi["x"], hi["dt"], hi["A"], hi["B"], hi["C"], hi["D"],
                              chunk_size=128, initial_state=hi["init"])
    torch.cuda.synchronize()
    assert torch.equal(fin, inp["init"])
    inp0 = case_inputs(1, 0, 2, 64, 64, 1, 128, init="zero", seed=2)
    hi0 = _pinned(inp0)
    _, fin0 = ssd.ssd_fwd_host(hi0["x"], hi0["dt"], hi0["A"], hi0["B"], hi0["C"], hi0["D"],
                               chunk_size=128)
    torch.cuda.synchronize()
    assert float(fin0.abs().max()) == 0.0
