"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times.

The GPU runs the whole problem (every batch row and head, the same
chunk_size and path the benchmark uses); the float64 oracle then recomputes
a sample of (batch row, head) pairs exactly.  Heads are independent given
their group's B and C, so a sample is checked element by element against the
oracle with no approximation: m heads are taken from each sampled group, and
the sampled problem has one group per sampled group (heads_per_group = m), so
every sampled head keeps its own B and C.

Workloads: the 2.7B-layer shape (B 4, L 4096, H 80, P 64, S 128, chunk 256),
the long grouped shape with an initial state (B 2, L 32768, H 64, S 256,
G 8), the extreme length with every chunk state (B 1, L 262144, H 32,
S 512, chunk 128) and every point of the length x dstate sweep (L 1K-256K
x S 64-512, 256K tokens) with the chunk size left to the library's tuner,
plus the ragged L = 4095.
"""
import pytest
import torch

import oracle
from parity_util import assert_parity, to_gpu
import state_space_sequence_cumsum_gb300 as ssd
from state_space_sequence_cumsum_gb300.inputs import (EXTREME_256K, LAYER_2P7B, LONG_S256_G8,
                                                      Shape, make_inputs, sweep_shape)

pytestmark = pytest.mark.gpu


def sample(inp, shape: Shape, batches, heads_per_group: dict):
    """CPU inputs restricted to the sampled batch rows and heads.

    heads_per_group maps a group index to the heads taken from it (the same
    count from every sampled group, so head k of the sample lies in sampled
    group k // m)."""
    hpg = shape.nheads // shape.ngroups
    groups = sorted(heads_per_group)
    m = len(heads_per_group[groups[0]])
    heads = []
    for gq in groups:
        hs = sorted(heads_per_group[gq])
        assert len(hs) == m and all(h // hpg == gq for h in hs)
        heads += hs
    b = torch.tensor(batches)
    h = torch.tensor(heads)
    gidx = torch.tensor(groups)
    sub = {
        "x": inp["x"][b][:, :, h], "dt": inp["dt"][b][:, :, h], "A": inp["A"][h],
        "B": inp["B"][b][:, :, gidx], "C": inp["C"][b][:, :, gidx], "D": inp["D"][h],
        "init": None if inp["init"] is None else inp["init"][b][:, h],
    }
    return sub, b, h


def run_full(shape: Shape, dtype, init, want_states, chunk_size, batches, heads_per_group):
    inp = make_inputs(shape, dtype=dtype, init=init, seed=0)
    g = to_gpu(inp)
    y, fin, st = ssd.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"],
                             chunk_size=chunk_size, initial_state=g["init"],
                             return_final_state=True, return_chunk_states=want_states)
    torch.cuda.synchronize()
    assert ssd.ssd_stream_status() == 0
    sub, b, h = sample(inp, shape, batches, heads_per_group)
    T = chunk_size or ssd.ssd_fwd_chosen_chunk_size(shape.batch, shape.seqlen, shape.nheads,
                                                    shape.headdim, shape.dstate, shape.ngroups,
                                                    dtype)
    ref = oracle.fwd(sub["x"], sub["dt"], sub["A"], sub["B"], sub["C"], sub["D"], T,
                     init=sub["init"], want_states=want_states)
    bd, hd = b.to(y.device), h.to(y.device)
    assert_parity(y.index_select(0, bd).index_select(2, hd), ref["y"], dtype, "y")
    assert_parity(fin.index_select(0, bd).index_select(1, hd), ref["final_state"], dtype,
                  "final_state")
    if want_states:
        assert_parity(st.index_select(0, bd).index_select(1, hd), ref["chunk_states"], dtype,
                      "chunk_states")
    return T


def test_layer_2p7b_shape():
    """B 4, L 4096, H 80, P 64, S 128, G 1, chunk 256, bf16, zero init, final state."""
    run_full(LAYER_2P7B, torch.bfloat16, "zero", False, 256, [0, 3],
             {0: [0, 13, 29, 41, 58, 79]})


def test_long_grouped_with_initial_state():
    """B 2, L 32768, H 64, P 64, S 256, G 8, chunk 256, bf16, N(0, 0.1) init."""
    run_full(LONG_S256_G8, torch.bfloat16, "randn", False, 256, [0, 1],
             {0: [0, 5], 3: [24, 30], 7: [57, 63]})


def test_extreme_length_all_chunk_states():
    """B 1, L 262144, H 32, P 64, S 512, G 1, chunk 128, bf16, every chunk state."""
    run_full(EXTREME_256K, torch.bfloat16, "zero", True, 128, [0], {0: [0, 15, 31]})


def sweep_sample(L: int, batch: int):
    """Sampled (batch rows, heads) of one sweep point: about 256K-512K
    sampled token-heads per point, first and last rows included."""
    if L >= 65536:
        return [batch - 1], [3, 60]
    if L >= 16384:
        return [1, batch - 1], [5, 50]
    if L >= 4095:
        return [0, batch // 2, batch - 1], [0, 31, 63]
    return [0, 100, batch - 1], [7, 42, 63]


SWEEP = [(L, S) for L in (1024, 4096, 16384, 65536, 262144) for S in (64, 128, 256, 512)]
SWEEP.append((4095, 128))  # ragged last chunk, B 64


@pytest.mark.parametrize("L,S", SWEEP, ids=[f"L{L}-S{S}" for L, S in SWEEP])
def test_length_dstate_sweep(L, S):
    """batch x L = 256K tokens, 64 heads, P 64, G 1, bf16; chunk size left to
    the library (chunk_size 0), which times {64, 128, 256} on this very call
    and keeps the fastest -- the launch configuration the benchmark times."""
    shape = sweep_shape(L, S, 0)
    batches, heads = sweep_sample(L, shape.batch)
    T = run_full(shape, torch.bfloat16, "zero", False, 0, batches, {0: heads})
    assert T in (64, 128, 256)
    assert ssd.ssd_fwd_chunk_size_was_timed(shape.batch, L, 64, 64, S, 1, torch.bfloat16)
