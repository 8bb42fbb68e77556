"""Failure detection without a GPU fault.

Every wait in the kernels is bounded: when one runs out, the kernel records
the error in the library's per-device status word, every role leaves its
loop with no copy or MMA in flight, TMEM is freed, and the host reads
SSD_ERR_TIMEOUT from ssd_stream_status.  The test makes a wait run out on
purpose with the library's host-set debug parameter SSD_FAULT_SKIP_ARRIVE=1:
one compute warp of the head-pair kernel skips its barrier arrival on the
first tile (a barrier that nothing else will complete) and the waits are
shortened to 20 ms.  Nothing traps or hangs; the next call runs normally.
"""
import pytest
import torch

from parity_util import assert_parity, case_inputs, oracle_run, to_gpu
import state_space_sequence_cumsum_gb300 as ssd
from state_space_sequence_cumsum_gb300 import _lib

pytestmark = pytest.mark.gpu


def test_lost_arrival_reports_timeout_then_next_call_is_clean(monkeypatch):
    # one 128-token tile, one head pair: one CTA, one item
    inp = case_inputs(1, 128, 2, 64, 128, 1, 128, seed=41)
    g = to_gpu(inp)
    args = (g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"])
    assert ssd.ssd_fwd_path(g["x"], g["B"], 128) == "fused-pair-tensor-cores"
    assert ssd.ssd_stream_status() == _lib.SSD_OK
    monkeypatch.setenv("SSD_FAULT_SKIP_ARRIVE", "1")
    ssd.ssd_fwd(*args, chunk_size=128)
    assert ssd.ssd_stream_status() == _lib.SSD_ERR_TIMEOUT
    # reading the status cleared it
    assert ssd.ssd_stream_status() == _lib.SSD_OK
    monkeypatch.delenv("SSD_FAULT_SKIP_ARRIVE")
    y, fin, _ = ssd.ssd_fwd(*args, chunk_size=128)
    assert ssd.ssd_stream_status() == _lib.SSD_OK
    ref = oracle_run(inp, 128)
    assert_parity(y, ref["y"], torch.bfloat16, "y after the injected timeout")
    assert_parity(fin, ref["final_state"], torch.bfloat16, "final_state after the injected timeout")
