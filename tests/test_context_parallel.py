"""Sequence-sharded (context-parallel) forward.

Section "Kernel 2: fwd_pass_state" of the cuTile Mamba-2 post makes the state
at the end of one call the initial state of the next, and the state update
is linear in the state.  So a sequence cut into R segments runs as: every
segment from a zero state (end state s_k, total decay D_k), one exchange of
(s_k, D_k), the carried-in state h_r = exp2(D_{r-1}) h_{r-1} + s_{r-1}, and
every segment's forward from h_r.  The result must equal the unsharded run:
here, the oracle's token recurrence over the whole sequence.

* CPU (no GPU): the host logic of ssd_fwd_context_parallel under two gloo
  ranks -- which rank sends what, the order of the gathered summaries and
  the carried-in state each rank starts from -- with the three library
  calls replaced by float64 stand-ins written here.
* GPU: ssd_segment_summary and ssd_carry_in against the oracle; R segments
  run one after another in one process through the C ABI; and two processes
  on the one GPU exchanging their summaries over gloo (no kernel waits on
  another process).
"""
import math
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))
for p_ in (ROOT, TESTS):
    if p_ not in sys.path:
        sys.path.insert(0, p_)

import oracle  # noqa: E402
from parity_util import assert_parity, case_inputs, to_gpu  # noqa: E402

LOG2E = 1.0 / math.log(2.0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _segments(L, R, T):
    """R contiguous segments of whole chunks (the last one takes the rest)."""
    per = (L + R - 1) // R
    per = (per + T - 1) // T * T
    cuts = [min(L, k * per) for k in range(R + 1)]
    cuts[-1] = L
    return list(zip(cuts[:-1], cuts[1:]))


def _slice(inp, a, b):
    return {k: (v[:, a:b].contiguous() if k in ("x", "dt", "B", "C") else v)
            for k, v in inp.items()}


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


# ------------------------------------------------------------------ CPU: host logic

def _install_stand_ins(ssd):
    """float64 stand-ins for the three library calls, so the orchestration
    runs on the CPU: the oracle's recurrence for the runs, the closed form
    sum of A dt for the decay, and the carry written out."""
    def summary(x, dt, A, B, chunk_size, workspace=None, stream=None):
        H = x.shape[2]
        ref = oracle.fwd(x, dt, A, B, B, torch.zeros(H), chunk_size)
        dec = LOG2E * (_np(dt) * _np(A)[None, None, :]).sum(axis=1)
        return torch.from_numpy(ref["final_state"]).float(), torch.from_numpy(dec).float()

    def carry_in(seg_states, seg_decays, upto, initial_state=None, out=None, stream=None):
        s, d = _np(seg_states), _np(seg_decays)
        h = np.zeros(s.shape[1:]) if initial_state is None else _np(initial_state)
        for k in range(upto):
            h = np.exp2(d[k])[:, :, None, None] * h + s[k]
        return torch.from_numpy(h).float()

    def fwd(x, dt, A, B, C, D, chunk_size=0, initial_state=None, return_final_state=True,
            return_chunk_states=False, workspace=None, stream=None):
        ref = oracle.fwd(x, dt, A, B, C, D, chunk_size, init=initial_state,
                         want_states=return_chunk_states)
        st = torch.from_numpy(ref["chunk_states"]) if return_chunk_states else None
        return torch.from_numpy(ref["y"]), torch.from_numpy(ref["final_state"]), st

    ssd.ssd_segment_summary = summary
    ssd.ssd_carry_in = carry_in
    ssd.ssd_fwd = fwd


def _cpu_worker(rank, ws, port, shape, cuts, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    from state_space_sequence_cumsum_gb300 import ssd
    _install_stand_ins(ssd)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        inp = case_inputs(*shape, init="randn", seed=5)
        a, b = cuts[rank]
        seg = _slice(inp, a, b)
        y, fin, st = ssd.ssd_fwd_context_parallel(seg["x"], seg["dt"], seg["A"], seg["B"],
                                                  seg["C"], seg["D"], shape[6],
                                                  initial_state=inp["init"],
                                                  return_chunk_states=True)
        out[rank] = (y.numpy(), fin.numpy(), st.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("ws", [2, 3])
def test_host_logic_under_gloo_ranks_equals_one_run(ws):
    shape = (2, 200, 4, 8, 8, 2, 16)  # B, L, H, P, S, G, T
    cuts = _segments(shape[1], ws, shape[6])
    port = _free_port()
    # the manager process is started by spawn too: never fork a process
    # that may hold a CUDA context
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_cpu_worker, args=(ws, port, shape, cuts, out), nprocs=ws, join=True)
        res = dict(out)
    inp = case_inputs(*shape, init="randn", seed=5)
    ref = oracle.fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], shape[6],
                     init=inp["init"], want_states=True)
    y = np.concatenate([res[r][0] for r in range(ws)], axis=1)
    st = np.concatenate([res[r][2] for r in range(ws)], axis=2)
    # the summaries cross the exchange as f32: agreement to f32 rounding
    np.testing.assert_allclose(y, ref["y"], rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(st, ref["chunk_states"], rtol=1e-5, atol=1e-5)
    # the last segment's final state is the sequence's
    np.testing.assert_allclose(res[ws - 1][1], ref["final_state"], rtol=1e-5, atol=1e-5)


# ------------------------------------------------------------------ GPU

def _run_segments(inp, T, R, dtype):
    """R segments run one after another in this process through the C ABI."""
    import state_space_sequence_cumsum_gb300 as ssd
    g = to_gpu(inp)
    L = inp["x"].shape[1]
    cuts = _segments(L, R, T)
    summ = []
    for (a, b) in cuts:
        s = _slice(g, a, b)
        summ.append(ssd.ssd_segment_summary(s["x"], s["dt"], s["A"], s["B"], T))
    seg_states = torch.stack([s for s, _ in summ])
    seg_decays = torch.stack([d for _, d in summ])
    ys, sts, fin = [], [], None
    for r, (a, b) in enumerate(cuts):
        s = _slice(g, a, b)
        h_in = ssd.ssd_carry_in(seg_states, seg_decays, r, initial_state=g["init"])
        y, fin, st = ssd.ssd_fwd(s["x"], s["dt"], s["A"], s["B"], s["C"], s["D"], chunk_size=T,
                                 initial_state=h_in, return_chunk_states=True)
        ys.append(y)
        sts.append(st)
    torch.cuda.synchronize()
    assert ssd.ssd_stream_status() == 0
    return torch.cat(ys, dim=1), fin, torch.cat(sts, dim=2)


@pytest.mark.gpu
@pytest.mark.parametrize("B,L,H,P,S,G,T,dtype,R", [
    (2, 1024, 4, 64, 128, 1, 128, torch.bfloat16, 4),    # head-pair path
    (1, 1000, 6, 64, 64, 3, 128, torch.bfloat16, 3),     # ragged last segment
    (1, 2048, 4, 64, 256, 2, 256, torch.bfloat16, 2),    # one-head fused path
    (1, 768, 2, 64, 512, 1, 128, torch.bfloat16, 3),     # staged, dstate 512 (chunk states)
    (2, 333, 3, 32, 48, 1, 64, torch.float32, 3),        # f32 CUDA cores
])
def test_segments_in_sequence_equal_one_run(B, L, H, P, S, G, T, dtype, R):
    inp = case_inputs(B, L, H, P, S, G, T, dtype=dtype, init="randn", seed=7)
    y, fin, st = _run_segments(inp, T, R, dtype)
    ref = oracle.fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], T,
                     init=inp["init"], want_states=True)
    assert_parity(y, ref["y"], dtype, "y")
    assert_parity(fin, ref["final_state"], dtype, "final_state")
    assert_parity(st, ref["chunk_states"], dtype, "chunk_states")


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_segment_summary_and_carry_in(dtype):
    import state_space_sequence_cumsum_gb300 as ssd
    B, L, H, P, S, G, T = 2, 600, 4, 64, 128, 2, 128
    inp = case_inputs(B, L, H, P, S, G, T, dtype=dtype, init="randn", seed=9)
    g = to_gpu(inp)
    st, dec = ssd.ssd_segment_summary(g["x"], g["dt"], g["A"], g["B"], T)
    ref = oracle.fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], T)
    assert_parity(st, ref["final_state"], dtype, "segment end state from zero")
    want = LOG2E * (_np(inp["dt"]) * _np(inp["A"])[None, None, :]).sum(axis=1)
    np.testing.assert_allclose(_np(dec), want, rtol=1e-5, atol=1e-5 * np.abs(want).max())
    # carry-in over three made-up segment summaries, written out in float64
    gen = torch.Generator().manual_seed(3)
    ss = torch.randn((3, B, H, P, S), generator=gen)
    dd = -torch.rand((3, B, H), generator=gen) * 4
    h0 = inp["init"]
    h = _np(h0)
    for upto in range(4):
        got = ssd.ssd_carry_in(ss.cuda(), dd.cuda(), upto, initial_state=h0.cuda())
        np.testing.assert_allclose(_np(got), h, rtol=1e-5, atol=1e-5)
        if upto < 3:
            h = np.exp2(_np(dd[upto]))[:, :, None, None] * h + _np(ss[upto])
    zero = ssd.ssd_carry_in(ss.cuda(), dd.cuda(), 0)
    assert torch.count_nonzero(zero) == 0


def _gpu_worker(rank, ws, port, shape, cuts, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import state_space_sequence_cumsum_gb300 as ssd
    torch.cuda.set_device(0)  # both processes share the one GPU
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        inp = case_inputs(*shape, init="randn", seed=11)
        a, b = cuts[rank]
        seg = to_gpu(_slice(inp, a, b))
        y, fin, st = ssd.ssd_fwd_context_parallel(seg["x"], seg["dt"], seg["A"], seg["B"],
                                                  seg["C"], seg["D"], shape[6],
                                                  initial_state=seg["init"],
                                                  return_chunk_states=True)
        torch.cuda.synchronize()
        out[rank] = (_np(y), _np(fin), _np(st), int(ssd.ssd_stream_status()))
    finally:
        dist.destroy_process_group()


@pytest.mark.gpu
def test_two_processes_on_one_gpu_over_gloo():
    shape = (2, 1536, 4, 64, 128, 1, 256)  # B, L, H, P, S, G, T
    ws = 2
    cuts = _segments(shape[1], ws, shape[6])
    port = _free_port()
    # the manager process is started by spawn too: never fork a process
    # that may hold a CUDA context
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_gpu_worker, args=(ws, port, shape, cuts, out), nprocs=ws, join=True)
        res = dict(out)
    assert all(res[r][3] == 0 for r in range(ws))
    inp = case_inputs(*shape, init="randn", seed=11)
    ref = oracle.fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], shape[6],
                     init=inp["init"], want_states=True)
    y = np.concatenate([res[r][0] for r in range(ws)], axis=1)
    st = np.concatenate([res[r][2] for r in range(ws)], axis=2)
    assert_parity(torch.from_numpy(y), ref["y"], torch.bfloat16, "y")
    assert_parity(torch.from_numpy(st), ref["chunk_states"], torch.bfloat16, "chunk_states")
    assert_parity(torch.from_numpy(res[ws - 1][1]), ref["final_state"], torch.bfloat16,
                  "final_state")
