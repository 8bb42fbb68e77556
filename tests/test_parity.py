"""GPU parity of ssd_fwd (through the C ABI) against the float64 oracle.

Sizes here finish in seconds on the oracle yet span several tiles and a
ragged tail; edge cases cover empty, single-token, sub-chunk and
chunk-plus-one sequences, grouped B/C, an initial state, every supported
chunk size and the f32 path.  The full-size workloads are in
test_parity_full.py.
"""
import numpy as np
import pytest
import torch

from parity_util import TOL, assert_parity, case_inputs, oracle_run, to_gpu
import state_space_sequence_cumsum_gb300 as ssd

pytestmark = pytest.mark.gpu


def run_fwd(inp, T, want_states=True):
    g = to_gpu(inp)
    y, fin, st = ssd.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=T,
                             initial_state=g["init"], return_final_state=True,
                             return_chunk_states=want_states)
    assert ssd.ssd_stream_status() == 0
    return y, fin, st


def check_case(B, L, H, P, S, G, T, dtype, init="zero", seed=0, want_states=True):
    inp = case_inputs(B, L, H, P, S, G, T, dtype=dtype, init=init, seed=seed)
    y, fin, st = run_fwd(inp, T, want_states)
    ref = oracle_run(inp, T, want_states=want_states)
    assert_parity(y, ref["y"], dtype, "y")
    assert_parity(fin, ref["final_state"], dtype, "final_state")
    if want_states:
        assert_parity(st, ref["chunk_states"], dtype, "chunk_states")


def test_tiny_fp32_config():
    """batch 1, L 256, 2 heads, P 16, S 16, chunk 64, f32, zero init."""
    check_case(1, 256, 2, 16, 16, 1, 64, torch.float32)


@pytest.mark.parametrize("T", [64, 128, 256])
def test_bf16_chunk_sizes(T):
    check_case(2, 3 * T + 17, 4, 64, 128, 1, T, torch.bfloat16, init="randn", seed=T)


@pytest.mark.parametrize("P,S", [(32, 64), (64, 256), (128, 128), (64, 512), (16, 16)])
def test_bf16_head_and_state_sizes(P, S):
    check_case(1, 700, 4, P, S, 2, 128, torch.bfloat16, init="randn", seed=P + S)


@pytest.mark.parametrize("L", [1, 63, 64, 65, 129])
def test_edge_lengths(L):
    check_case(2, L, 4, 64, 128, 1, 64, torch.bfloat16, init="randn", seed=L)


@pytest.mark.parametrize("L", [1, 127, 128, 129, 255, 257])
def test_edge_lengths_tensor_core_tiles(L):
    check_case(2, L, 4, 64, 128, 1, 128, torch.bfloat16, init="randn", seed=L)
    check_case(1, L, 2, 64, 128, 1, 256, torch.bfloat16, init="randn", seed=L + 1)


@pytest.mark.parametrize("T", [128, 256])
def test_staged_tensor_core_path_matches_oracle(T, monkeypatch):
    """SSD_FWD_PATH=staged forces cumsum -> tcgen05 state pass -> tcgen05 chunk out."""
    monkeypatch.setenv("SSD_FWD_PATH", "staged")
    inp = case_inputs(2, 3 * T + 5, 4, 64, 128, 2, T, init="randn", seed=31)
    g = to_gpu(inp)
    assert ssd.ssd_fwd_path(g["x"], g["B"], T) == "staged-tensor-cores"
    check_case(2, 3 * T + 5, 4, 64, 128, 2, T, torch.bfloat16, init="randn", seed=31)


def test_fused_and_staged_paths_agree(monkeypatch):
    inp = case_inputs(1, 1000, 8, 64, 128, 1, 256, init="randn", seed=37)
    g = to_gpu(inp)
    assert ssd.ssd_fwd_path(g["x"], g["B"], 256) == "fused-pair-tensor-cores"
    y_f, f_f, _ = ssd.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], 256,
                              initial_state=g["init"])
    monkeypatch.setenv("SSD_FWD_PATH", "staged")
    y_s, f_s, _ = ssd.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], 256,
                              initial_state=g["init"])
    ref = oracle_run(inp, 256)
    assert_parity(y_f, ref["y"], torch.bfloat16, "fused y")
    assert_parity(y_s, ref["y"], torch.bfloat16, "staged y")
    assert_parity(f_f, ref["final_state"], torch.bfloat16, "fused final")
    assert_parity(f_s, ref["final_state"], torch.bfloat16, "staged final")


def test_empty_sequence_copies_init():
    inp = case_inputs(2, 0, 4, 64, 128, 1, 64, init="randn", seed=5)
    y, fin, st = run_fwd(inp, 64)
    assert y.numel() == 0 and st.shape[2] == 0
    assert torch.equal(fin.cpu(), inp["init"])


def test_grouped_heads_share_B_and_C():
    check_case(2, 515, 8, 64, 128, 4, 128, torch.bfloat16, init="randn", seed=9)


def test_fp32_path_several_tiles():
    check_case(2, 333, 3, 64, 96, 3, 64, torch.float32, init="randn", seed=11)


def test_auto_chunk_size_and_no_states():
    inp = case_inputs(1, 1000, 4, 64, 128, 1, 64, seed=13)
    g = to_gpu(inp)
    y, fin, st = ssd.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=0)
    assert st is None
    T = ssd.ssd_fwd_chosen_chunk_size(1, 1000, 4, 64, 128, 1, torch.bfloat16)
    ref = oracle_run(inp, T)
    assert_parity(y, ref["y"], torch.bfloat16, "y")
    assert_parity(fin, ref["final_state"], torch.bfloat16, "final")


def test_auto_chunk_size_is_timed_then_fixed():
    """chunk_size 0: the first call without chunk states times the candidates
    {64, 128, 256} (section "Mamba-2 性能优化": the best configuration is
    searched per shape) and fixes the fastest; later calls, and calls that
    return chunk states, use that choice."""
    shape = (2, 1500, 6, 64, 128, 1, torch.bfloat16)  # a shape no other test uses
    inp = case_inputs(*shape[:6], 128, seed=23)
    g = to_gpu(inp)
    args = (g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"])
    assert not ssd.ssd_fwd_chunk_size_was_timed(*shape)
    y, fin, _ = ssd.ssd_fwd(*args, chunk_size=0)
    torch.cuda.synchronize()
    assert ssd.ssd_stream_status() == 0
    assert ssd.ssd_fwd_chunk_size_was_timed(*shape)
    T = ssd.ssd_fwd_chosen_chunk_size(*shape)
    assert T in (64, 128, 256)
    ref = oracle_run(inp, T, want_states=True)
    assert_parity(y, ref["y"], torch.bfloat16, "y")
    assert_parity(fin, ref["final_state"], torch.bfloat16, "final")
    y2, fin2, st = ssd.ssd_fwd(*args, chunk_size=0, return_chunk_states=True)
    assert ssd.ssd_fwd_chosen_chunk_size(*shape) == T
    assert st.shape[2] == (1500 + T - 1) // T
    assert_parity(y2, ref["y"], torch.bfloat16, "y (second call)")
    assert_parity(st, ref["chunk_states"], torch.bfloat16, "chunk_states")


def test_auto_chunk_size_with_chunk_states_first_keeps_the_static_choice():
    shape = (1, 900, 4, 64, 64, 2, torch.bfloat16)  # a shape no other test uses
    inp = case_inputs(*shape[:6], 128, init="randn", seed=29)
    g = to_gpu(inp)
    y, fin, st = ssd.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=0,
                             initial_state=g["init"], return_chunk_states=True)
    assert not ssd.ssd_fwd_chunk_size_was_timed(*shape)
    T = ssd.ssd_fwd_chosen_chunk_size(*shape)
    assert T == 128 and st.shape[2] == (900 + T - 1) // T
    ref = oracle_run(inp, T, want_states=True)
    assert_parity(y, ref["y"], torch.bfloat16, "y")
    assert_parity(st, ref["chunk_states"], torch.bfloat16, "chunk_states")
    # a later call without states does not re-time a fixed choice
    ssd.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=0,
                initial_state=g["init"])
    assert not ssd.ssd_fwd_chunk_size_was_timed(*shape)


def test_auto_chunk_size_f32_timed():
    shape = (1, 333, 3, 32, 48, 1, torch.float32)  # a shape no other test uses
    inp = case_inputs(*shape[:6], 64, dtype=torch.float32, init="randn", seed=31)
    g = to_gpu(inp)
    y, fin, _ = ssd.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=0,
                            initial_state=g["init"])
    assert ssd.ssd_fwd_chunk_size_was_timed(*shape)
    T = ssd.ssd_fwd_chosen_chunk_size(*shape)
    assert T in (64, 128, 256)
    ref = oracle_run(inp, T)
    assert_parity(y, ref["y"], torch.float32, "y")
    assert_parity(fin, ref["final_state"], torch.float32, "final")


def test_two_halves_with_carried_state_equal_one_run():
    """final_state of call 1 fed as init of call 2 reproduces the single run
    (section "Kernel 2": the final state is the next call's init_state)."""
    inp = case_inputs(2, 1024, 4, 64, 128, 1, 128, init="randn", seed=17)
    g = to_gpu(inp)
    y_full, f_full, _ = ssd.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], 128,
                                    initial_state=g["init"])
    cut = 384
    a = {k: (v[:, :cut].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in g.items()}
    b = {k: (v[:, cut:].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in g.items()}
    y1, f1, _ = ssd.ssd_fwd(a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], 128,
                            initial_state=a["init"])
    y2, f2, _ = ssd.ssd_fwd(b["x"], b["dt"], b["A"], b["B"], b["C"], b["D"], 128,
                            initial_state=f1)
    ref = oracle_run(inp, 128)
    assert_parity(torch.cat([y1, y2], dim=1), ref["y"], torch.bfloat16, "split y")
    assert_parity(f2, ref["final_state"], torch.bfloat16, "split final")
    assert_parity(y_full, ref["y"], torch.bfloat16, "full y")


def test_final_state_independent_of_chunk_size():
    inp = case_inputs(1, 777, 4, 64, 128, 1, 64, init="randn", seed=19)
    g = to_gpu(inp)
    finals = []
    for T in (64, 128, 256):
        _, f, _ = ssd.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], T,
                              initial_state=g["init"])
        finals.append(f)
    ref = oracle_run(inp, 64)["final_state"]
    for f in finals:
        assert_parity(f, ref, torch.bfloat16, "final")


def test_repeat_calls_are_deterministic():
    inp = case_inputs(1, 600, 4, 64, 128, 1, 128, seed=23)
    y1, f1, _ = run_fwd(inp, 128, False)
    y2, f2, _ = run_fwd(inp, 128, False)
    assert torch.equal(y1, y2) and torch.equal(f1, f2)


# ---- fused head-pair kernel: decay modes per head, segments, both kernels

def _decay_case(B, L, H, S, T, dts, As, seed):
    """Inputs whose heads have fixed dt and A, so each head's per-tile decay
    range log2(e) * |A| * dt * 128 is known: above 160 a head takes the exact
    per-element scores, at or below it the factorized form."""
    inp = case_inputs(B, L, H, 64, S, 1, T, init="randn", seed=seed)
    for h, (d, a) in enumerate(zip(dts, As)):
        inp["dt"][:, :, h] = d
        inp["A"][h] = a
    return inp


@pytest.mark.parametrize("kernel", ["pair", "single"])
def test_fused_kernels_every_decay_mode(kernel, monkeypatch):
    """Per-tile decay (log2 e |A| dt 128) by head: 1773, 3.7, 33, 1108, 2364,
    665, 148, 96.  Head pairs (0,1) exact+factorized, (2,3) factorized+exact,
    (4,5) exact+exact, (6,7) exact+factorized near the factorization limit;
    head 1 keeps its state scale for many tiles, head 2 folds it every few
    tiles, head 7 every tile.  Ragged length, init state, chunk states and
    final state."""
    if kernel == "single":
        monkeypatch.setenv("SSD_FUSED_KERNEL", "single")
    dts = [0.6, 0.01, 0.15, 0.5, 0.8, 0.4, 0.2, 0.13]
    As = [-16.0, -2.0, -1.2, -12.0, -16.0, -9.0, -4.0, -4.0]
    T = 256
    inp = _decay_case(2, 2000, 8, 128, T, dts, As, seed=41)
    y, fin, st = run_fwd(inp, T)
    ref = oracle_run(inp, T, want_states=True)
    assert_parity(y, ref["y"], torch.bfloat16, "y")
    assert_parity(fin, ref["final_state"], torch.bfloat16, "final_state")
    assert_parity(st, ref["chunk_states"], torch.bfloat16, "chunk_states")


@pytest.mark.parametrize("S", [64, 128])
@pytest.mark.parametrize("prefill", ["1", "0"])
def test_pair_kernel_many_segments(S, prefill, monkeypatch):
    """One batch row and four heads over 4095 tokens: the fused pass splits
    each sequence into many segments whose start states the segmented state
    pass computes beforehand (prefill), or, with that plan off, one CTA runs
    each head pair end to end."""
    monkeypatch.setenv("SSD_PAIR_PREFILL", prefill)
    check_case(1, 4095, 4, 64, S, 1, 128, torch.bfloat16, init="randn", seed=43 + S)


@pytest.mark.parametrize("T", [128, 256])
@pytest.mark.parametrize("init", ["zero", "randn"])
def test_pair_prefilled_segments_match_unsegmented(T, init, monkeypatch):
    """Few head pairs (one wave of (pair, segment) items): segments run at
    once from start states of the segmented state pass ("Kernel 2:
    fwd_pass_state" over parallel segments plus a serial combine).  The
    result matches the plan without segments (one CTA per head pair) and the
    oracle, chunk states included, over a ragged last segment and two tiles
    per chunk at T = 256."""
    inp = case_inputs(2, 3001, 4, 64, 128, 2, T, init=init, seed=T + 5)
    ref = oracle_run(inp, T, want_states=True)
    out = {}
    for mode in ("1", "0"):
        monkeypatch.setenv("SSD_PAIR_PREFILL", mode)
        out[mode] = run_fwd(inp, T)
        y, fin, st = out[mode]
        assert_parity(y, ref["y"], torch.bfloat16, "y")
        assert_parity(fin, ref["final_state"], torch.bfloat16, "final_state")
        assert_parity(st, ref["chunk_states"], torch.bfloat16, "chunk_states")
    scale = max(1.0, out["0"][1].abs().max().item())
    assert (out["1"][1] - out["0"][1]).abs().max().item() <= 1e-3 * scale


def test_pair_and_single_kernels_agree(monkeypatch):
    inp = case_inputs(2, 2000, 6, 64, 128, 3, 256, init="randn", seed=47)
    g = to_gpu(inp)
    y_p, f_p, _ = ssd.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], 256,
                              initial_state=g["init"])
    monkeypatch.setenv("SSD_FUSED_KERNEL", "single")
    y_s, f_s, _ = ssd.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], 256,
                              initial_state=g["init"])
    ref = oracle_run(inp, 256)
    for y, f, nm in ((y_p, f_p, "pair"), (y_s, f_s, "single")):
        assert_parity(y, ref["y"], torch.bfloat16, nm + " y")
        assert_parity(f, ref["final_state"], torch.bfloat16, nm + " final")


def test_pair_kernel_fast_decay_with_noise():
    """A head whose per-tile decay range is 130-190 (log2) with per-token dt
    noise, next to an ordinary head, over 64 tiles: each tile folds the
    state's scale at a reference far from the previous one, so two scale
    factors near 2^-75 meet (their product is below the f32 range)."""
    inp = case_inputs(1, 8192, 2, 64, 128, 1, 128, init="randn", seed=53)
    gen = torch.Generator().manual_seed(53)
    noise = torch.randn(1, 8192, generator=gen)
    inp["dt"][:, :, 0] = 0.06 * torch.exp(0.15 * noise)
    inp["A"][0] = -14.0
    y, fin, _ = run_fwd(inp, 128, want_states=False)
    ref = oracle_run(inp, 128)
    assert_parity(y, ref["y"], torch.bfloat16, "y")
    assert_parity(fin, ref["final_state"], torch.bfloat16, "final_state")


def test_pair_kernel_runs_with_the_smaller_workspace():
    """ssd_fwd_workspace_size reports the prefilled plan's workspace (it also
    holds G and dt^T); the head-pair path accepts less -- down to what the
    plan without segments needs -- and then runs that plan.  Found by
    bisection on the host-side check (a short workspace returns
    SSD_ERR_WORKSPACE before any launch), then run at exactly that size
    against the oracle."""
    import ctypes
    from state_space_sequence_cumsum_gb300 import _lib
    B, L, H, P, S, G, T = 1, 4095, 4, 64, 128, 1, 128
    inp = case_inputs(B, L, H, P, S, G, T, init="randn", seed=77)
    g = to_gpu(inp)
    lib = _lib.load()
    d = _lib.dims(B, L, H, P, S, G)
    pref = int(lib.ssd_fwd_workspace_size(d, 0, T, 0))
    big = torch.empty(pref, dtype=torch.uint8, device="cuda")
    y = torch.empty_like(g["x"])
    fin = torch.empty((B, H, P, S), device="cuda")
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call(nbytes):
        return lib.ssd_fwd(ptr(g["x"]), ptr(g["dt"]), ptr(g["A"]), ptr(g["B"]), ptr(g["C"]),
                           ptr(g["D"]), ptr(g["init"]), ptr(y), ptr(fin), None, d, 0, T,
                           ptr(big), ctypes.c_size_t(nbytes), stream)
    lo, hi = 0, pref // 256  # in 256-byte units: lo fails, hi works
    while hi - lo > 1:
        mid = (lo + hi) // 2
        st = call(mid * 256) if mid else _lib.SSD_ERR_WORKSPACE
        if st == _lib.SSD_OK:
            hi = mid
        else:
            assert st == _lib.SSD_ERR_WORKSPACE
            lo = mid
    least = hi * 256
    assert least < pref  # the plan without segments needs no G / dt^T copy
    assert call(least) == _lib.SSD_OK
    torch.cuda.synchronize()
    assert ssd.ssd_stream_status() == 0
    ref = oracle_run(inp, T)
    assert_parity(y, ref["y"], torch.bfloat16, "y")
    assert_parity(fin, ref["final_state"], torch.bfloat16, "final_state")
