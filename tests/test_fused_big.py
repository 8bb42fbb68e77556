"""GPU parity of the fused forward for dstate 384 / 512 against the float64 oracle.

At these state sizes one tile's B and C do not fit in shared memory next to
x, X_hat and H, so the fused kernel streams them in 128-row dstate blocks and
builds H one block at a time; the state stays in TMEM from tile to tile.
The cases cover each work plan the fused pass picks (prefilled segments for
few sequences, one CTA per sequence, segments that hand their states on when
there are more sequences than SMs), two tiles per chunk, ragged lengths, an
initial state with every chunk state and the final state returned, heads
whose decay over a tile is too wide for the factorized form (the exact
per-element scores), the stage-level entry point, and agreement with the
staged path.  Cases with many sequences check sampled heads (one head per
group, so the oracle runs on those heads alone).  With every chunk state
asked for, ssd_fwd takes the staged path at these state sizes;
SSD_FWD_PATH=fused keeps the fused kernel for those cases.
"""
import pytest
import torch

from parity_util import assert_parity, case_inputs, oracle_run, to_gpu
import state_space_sequence_cumsum_gb300 as ssd

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def fused_path(monkeypatch):
    monkeypatch.setenv("SSD_FWD_PATH", "fused")


def fwd(g, T, want_states=True):
    y, fin, st = ssd.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=T,
                             initial_state=g["init"], return_final_state=True,
                             return_chunk_states=want_states)
    assert ssd.ssd_stream_status() == 0
    return y, fin, st


def check(inp, T, heads=None, want_states=True):
    g = to_gpu(inp)
    assert ssd.ssd_fwd_path(g["x"], g["B"], T, want_states) == "fused-tensor-cores"
    y, fin, st = fwd(g, T, want_states)
    ref = oracle_run(inp, T, want_states=want_states, heads=heads)
    idx = torch.tensor(ref["heads"]) if heads is not None else None
    pick = (lambda t, d: t.index_select(d, idx.to(t.device))) if idx is not None else (lambda t, d: t)
    assert_parity(pick(y, 2), ref["y"], torch.bfloat16, "y")
    assert_parity(pick(fin, 1), ref["final_state"], torch.bfloat16, "final_state")
    if want_states:
        assert_parity(pick(st, 1), ref["chunk_states"], torch.bfloat16, "chunk_states")


def test_dstate_512_path_choice(monkeypatch):
    monkeypatch.delenv("SSD_FWD_PATH")
    inp = case_inputs(1, 300, 2, 64, 512, 1, 128)
    g = to_gpu(inp)
    assert ssd.ssd_fwd_path(g["x"], g["B"], 128) == "fused-tensor-cores"
    assert ssd.ssd_fwd_path(g["x"], g["B"], 256) == "fused-tensor-cores"
    # every chunk state asked for: the staged path
    assert ssd.ssd_fwd_path(g["x"], g["B"], 128, True) == "staged-tensor-cores"
    # 64-token chunks are not whole tiles: a staged path
    assert ssd.ssd_fwd_path(g["x"], g["B"], 64).startswith("staged-")


@pytest.mark.parametrize("B,L,H,P,S,G,T", [
    (1, 1000, 4, 64, 512, 2, 128),   # few sequences: prefilled segments
    (1, 1000, 3, 64, 384, 1, 256),   # dstate 384, two tiles per chunk
    (2, 645, 2, 64, 512, 1, 128),    # ragged tail
    (1, 129, 2, 64, 512, 1, 128),    # two tiles, one CTA per sequence
    (1, 1, 2, 64, 512, 1, 128),      # a single token
])
def test_fused_dstate_blocks_match_oracle(B, L, H, P, S, G, T):
    check(case_inputs(B, L, H, P, S, G, T, init="randn", seed=L + S + H), T)


def test_one_cta_per_sequence_plan():
    """100 sequences: more than half the SMs, so no state pass; each CTA runs
    its sequence end to end."""
    inp = case_inputs(1, 300, 100, 64, 512, 100, 128, init="randn", seed=41)
    check(inp, 128, heads=[0, 37, 99])


def test_hand_off_segments_plan():
    """160 sequences, more than the SMs: segments hand their states on."""
    inp = case_inputs(2, 300, 80, 64, 512, 80, 128, init="randn", seed=43)
    check(inp, 128, heads=[1, 40, 79])


def test_fast_decaying_heads_take_the_exact_form():
    """dt twenty times larger on two heads: their tiles' decay ranges exceed
    the factorized form's bound, so their scores are exact per element (and
    their Y1 goes through the CB columns); the other heads stay factorized."""
    inp = case_inputs(1, 700, 4, 64, 512, 2, 128, init="randn", seed=47)
    inp["dt"] = inp["dt"].clone()
    inp["dt"][:, :, :2] *= 20.0
    check(inp, 128)


def test_without_chunk_states():
    check(case_inputs(1, 520, 2, 64, 512, 1, 128, init="randn", seed=53), 128, want_states=False)


def test_fused_and_staged_agree(monkeypatch):
    inp = case_inputs(1, 777, 2, 64, 512, 1, 128, init="randn", seed=59)
    g = to_gpu(inp)
    y_f, f_f, s_f = fwd(g, 128)
    monkeypatch.setenv("SSD_FWD_PATH", "staged")
    assert ssd.ssd_fwd_path(g["x"], g["B"], 128) == "staged-tensor-cores"
    y_s, f_s, s_s = fwd(g, 128)
    ref = oracle_run(inp, 128, want_states=True)
    for what, a, b, r in (("y", y_f, y_s, ref["y"]), ("final_state", f_f, f_s, ref["final_state"]),
                          ("chunk_states", s_f, s_s, ref["chunk_states"])):
        assert_parity(a, r, torch.bfloat16, "fused " + what)
        assert_parity(b, r, torch.bfloat16, "staged " + what)


def test_state_out_entry_point():
    """ssd_state_out (stages 2 + 3 fused, from G and dt^T) at dstate 512: it
    always runs the fused kernel, chunk states or not."""
    inp = case_inputs(1, 600, 2, 64, 512, 1, 128, init="randn", seed=61)
    g = to_gpu(inp)
    Gc, dtT = ssd.ssd_chunk_cumsum(g["dt"], g["A"], 128)
    y, fin, st = ssd.ssd_state_out(g["x"], g["B"], g["C"], dtT, Gc, g["D"], 128,
                                   initial_state=g["init"], chunk_states=True)
    assert ssd.ssd_stream_status() == 0
    ref = oracle_run(inp, 128, want_states=True)
    assert_parity(y, ref["y"], torch.bfloat16, "y")
    assert_parity(fin, ref["final_state"], torch.bfloat16, "final_state")
    assert_parity(st, ref["chunk_states"], torch.bfloat16, "chunk_states")
