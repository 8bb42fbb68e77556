"""Pins for the float64 oracle (CPU only).

Every check here compares the oracle's token recurrence with something other
than itself: hand-worked golden values, the fully unrolled quadratic form
(brute force), the pages' chunked closed form, the decay-free
linear-attention reduction, and invariants the mathematics fixes.  The
source is "Accelerating Mamba-2 forward-pass kernels with CUDA Tile
(cuTile)" (dbyun.net/article/14364), sections "Mamba-2 架构" (recurrence,
jump formula, linear-attention form, log-space unrolling, chunk output
equation), "Kernel 1" (within-chunk cumsum in log2 units) and "Kernel 2"
(chunk start states, final state, carry into the next call).
"""
import math
import os

import numpy as np
import pytest
import torch

from state_space_sequence_cumsum_gb300.inputs import Shape, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
LOG2E = 1.0 / math.log(2.0)


def _f64(t):
    return None if t is None else t.to(torch.float64).numpy()


def case(B, L, H, P, S, G, T, init="randn", seed=1, dtype=torch.float32):
    inp = make_inputs(Shape(B, L, H, P, S, G, T), dtype=dtype, init=init, seed=seed)
    return {k: _f64(v) for k, v in inp.items()}


def run(oracle, c, T, want_states=False, **over):
    d = dict(c)
    d.update(over)
    return oracle.fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], T, init=d["init"],
                      want_states=want_states)


# ---------------------------------------------------------------- independent forms

def brute_force(x, dt, A, Bm, Cm, D, h0):
    """Unrolled form of the recurrence (section "Mamba-2 架构", log-space unrolling):
    y_t = sum_{j<=t} exp(sum_{k=j+1}^{t} a_k) dt_j (C_t . B_j) x_j
          + exp(sum_{k<=t} a_k) h0 C_t + D x_t,   a_k = A dt_k.
    Plain loops; tiny inputs only."""
    B, L, H, P = x.shape
    G, S = Bm.shape[2], Bm.shape[3]
    hpg = H // G
    y = np.zeros_like(x)
    final = np.zeros((B, H, P, S))
    for b in range(B):
        for h in range(H):
            g = h // hpg
            csum = np.cumsum(A[h] * dt[b, :, h])
            for t in range(L):
                acc = np.zeros(P)
                for j in range(t + 1):
                    w = math.exp(csum[t] - csum[j]) * dt[b, j, h] * float(Cm[b, t, g] @ Bm[b, j, g])
                    acc += w * x[b, j, h]
                if h0 is not None:
                    acc += math.exp(csum[t]) * (h0[b, h] @ Cm[b, t, g])
                y[b, t, h] = acc + D[h] * x[b, t, h]
            for j in range(L):
                w = math.exp(csum[L - 1] - csum[j]) * dt[b, j, h]
                final[b, h] += w * np.outer(x[b, j, h], Bm[b, j, g])
            if h0 is not None and L > 0:
                final[b, h] += math.exp(csum[L - 1]) * h0[b, h]
    return y, final


def chunked_closed_form(x, dt, A, Bm, Cm, D, h0, T):
    """The pages' chunk equations in natural-log units:
    jump   h_{next} = exp(G_last) h + (exp(G_last - G) * dt * B)^T X   (as [P,S]: X^T (w*B))
    output Y = exp(G) (C h^T) + (exp(G_i - G_j) (C B^T) M) (dt X) + D X
    with G the within-chunk cumsum of a and G_last at the chunk's last valid token."""
    B, L, H, P = x.shape
    G, S = Bm.shape[2], Bm.shape[3]
    hpg = H // G
    nc = (L + T - 1) // T
    y = np.zeros_like(x)
    final = np.zeros((B, H, P, S))
    states = np.zeros((B, H, nc, P, S))
    for b in range(B):
        for h in range(H):
            g = h // hpg
            hs = np.zeros((P, S)) if h0 is None else h0[b, h].copy()
            for c in range(nc):
                sl = slice(c * T, min(L, (c + 1) * T))
                states[b, h, c] = hs
                Gc = np.cumsum(A[h] * dt[b, sl, h])
                X, Bc, Cc, dtc = x[b, sl, h], Bm[b, sl, g], Cm[b, sl, g], dt[b, sl, h]
                n = Gc.shape[0]
                causal = np.tril(np.ones((n, n), dtype=bool))
                decay = np.exp(np.where(causal, Gc[:, None] - Gc[None, :], -np.inf))
                scores = (Cc @ Bc.T) * decay
                y[b, sl, h] = (np.exp(Gc)[:, None] * (Cc @ hs.T) + scores @ (dtc[:, None] * X)
                               + D[h] * X)
                Glast = Gc[-1]
                hs = math.exp(Glast) * hs + X.T @ (Bc * (np.exp(Glast - Gc) * dtc)[:, None])
            final[b, h] = hs
    return y, final, states


def assert_close(a, b, rtol=1e-11, what=""):
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= rtol * scale, f"{what}: max abs err {err:.3e} > {rtol:.1e} * {scale:.3e}"


# ---------------------------------------------------------------- golden fixtures

def load_golden(name):
    vals, dims = {}, {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *rest = line.split()
            if key == "dims":
                for kv in rest:
                    k, v = kv.split("=")
                    dims[k] = int(v)
            else:
                vals[key] = np.array([float(v) for v in rest])
    return dims, vals


@pytest.mark.parametrize("name", ["scalar_three_tokens.txt", "matrix_state_two_tokens.txt"])
def test_golden_hand_worked(oracle_mod, name):
    d, v = load_golden(name)
    B, L, H, P, S, G, T = (d[k] for k in "B L H P S G T".split())
    nc = (L + T - 1) // T
    x = v["x"].reshape(B, L, H, P)
    dt = v["dt"].reshape(B, L, H)
    Bm = v["Bm"].reshape(B, L, G, S)
    Cm = v["Cm"].reshape(B, L, G, S)
    init = v["init"].reshape(B, H, P, S)
    out = oracle_mod.fwd(x, dt, v["A"], Bm, Cm, v["D"], T, init=init, want_states=True)
    assert_close(out["y"], v["y"].reshape(B, L, H, P), 1e-14, "y")
    assert_close(out["final_state"], v["final"].reshape(B, H, P, S), 1e-14, "final")
    assert_close(out["chunk_states"], v["states"].reshape(B, H, nc, P, S), 1e-14, "states")
    Gl = oracle_mod.chunk_cumsum(dt, v["A"], T)
    assert_close(Gl, v["Glog2"].reshape(B, H, L), 1e-14, "G")


# ---------------------------------------------------------------- P1 brute force

@pytest.mark.parametrize("dims", [(1, 1, 1, 1, 1, 1), (1, 9, 2, 3, 4, 1), (2, 17, 4, 4, 3, 2),
                                  (1, 33, 3, 2, 5, 3)])
@pytest.mark.parametrize("init", ["zero", "randn"])
def test_brute_force(oracle_mod, dims, init):
    B, L, H, P, S, G = dims
    c = case(B, L, H, P, S, G, 8, init=init, seed=L + H)
    out = run(oracle_mod, c, 8)
    y, final = brute_force(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], c["init"])
    assert_close(out["y"], y, 1e-12, "y")
    assert_close(out["final_state"], final, 1e-12, "final")


# ---------------------------------------------------------------- P2 chunked closed form

@pytest.mark.parametrize("T", [1, 7, 16, 64, 100])
def test_chunked_closed_form(oracle_mod, T):
    c = case(2, 100, 4, 8, 6, 2, T, init="randn", seed=T)
    out = run(oracle_mod, c, T, want_states=True)
    y, final, states = chunked_closed_form(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"],
                                           c["init"], T)
    assert_close(out["y"], y, 1e-11, "y")
    assert_close(out["final_state"], final, 1e-11, "final")
    assert_close(out["chunk_states"], states, 1e-11, "states")


# ---------------------------------------------------------------- P3 linear attention

def test_decay_free_is_linear_attention(oracle_mod):
    """A = 0, dt = 1: Y = ((C B^T) * M) X + C h0^T + D X (section "Mamba-2 架构",
    linear-attention form with the causal mask)."""
    c = case(1, 40, 2, 5, 7, 1, 16, init="randn", seed=3)
    c["A"] = np.zeros_like(c["A"])
    c["dt"] = np.ones_like(c["dt"])
    out = run(oracle_mod, c, 16)
    L = 40
    M = np.tril(np.ones((L, L)))
    for h in range(2):
        X, Bc, Cc = c["x"][0, :, h], c["B"][0, :, 0], c["C"][0, :, 0]
        Y = ((Cc @ Bc.T) * M) @ X + Cc @ c["init"][0, h].T + c["D"][h] * X
        assert_close(out["y"][0, :, h], Y, 1e-12, f"head {h}")


# ---------------------------------------------------------------- G (Kernel 1)

def test_chunk_cumsum_closed_forms(oracle_mod):
    B, L, H, T = 2, 70, 3, 16
    A = np.array([-1.0, -2.5, -16.0])
    dt = np.full((B, L, H), 0.125)
    G = oracle_mod.chunk_cumsum(dt, A, T)
    pos = (np.arange(L) % T) + 1  # restarts at each chunk
    expect = LOG2E * A[None, :, None] * 0.125 * pos[None, None, :]
    assert_close(G, np.broadcast_to(expect, G.shape), 1e-14, "constant dt")
    # the first token of every chunk is just log2e * a_t
    c = case(B, L, H, 4, 4, 1, T, seed=5)
    G = oracle_mod.chunk_cumsum(c["dt"], c["A"], T)
    first = np.arange(0, L, T)
    assert_close(G[:, :, first], LOG2E * c["A"][None, :, None] *
                 np.transpose(c["dt"], (0, 2, 1))[:, :, first], 1e-14, "chunk starts")


def test_G_matches_recurrence_decay(oracle_mod):
    """With B = 0 the state only decays: final = h0 * 2^(sum over chunks of G_last)."""
    B, L, H, P, S, T = 1, 50, 2, 3, 4, 16
    c = case(B, L, H, P, S, 1, T, init="randn", seed=7)
    out = run(oracle_mod, c, T, B=np.zeros_like(c["B"]))
    G = oracle_mod.chunk_cumsum(c["dt"], c["A"], T)
    last = [min(L, (k + 1) * T) - 1 for k in range((L + T - 1) // T)]
    total = G[:, :, last].sum(axis=-1)  # [B, H]
    assert_close(out["final_state"], c["init"] * np.exp2(total)[:, :, None, None], 1e-12)


# ---------------------------------------------------------------- P4 invariants

def test_final_state_independent_of_chunk_size(oracle_mod):
    c = case(1, 90, 2, 4, 4, 1, 8, seed=11)
    f = [run(oracle_mod, c, T)["final_state"] for T in (1, 16, 64, 90)]
    for other in f[1:]:
        assert_close(other, f[0], 1e-14)


@pytest.mark.parametrize("split", [32, 45])
def test_two_halves_with_carry_equal_full_run(oracle_mod, split):
    """Section "Kernel 2": the final state is the next call's init_state."""
    c = case(2, 96, 2, 4, 5, 1, 32, seed=13)
    full = run(oracle_mod, c, 32)
    first = {k: (v[:, :split] if k in ("x", "dt", "B", "C") else v) for k, v in c.items()}
    second = {k: (v[:, split:] if k in ("x", "dt", "B", "C") else v) for k, v in c.items()}
    o1 = run(oracle_mod, first, 32)
    second["init"] = o1["final_state"]
    o2 = run(oracle_mod, second, 32)
    assert_close(np.concatenate([o1["y"], o2["y"]], axis=1), full["y"], 1e-12, "y")
    assert_close(o2["final_state"], full["final_state"], 1e-12, "final")


def test_token_by_token_with_carry_equals_full_run(oracle_mod):
    """The decode step's reference: L one-token calls, each starting from the
    previous call's final state, reproduce one L-token call (section
    "Mamba-2 架构": the recurrence needs nothing but the carried state)."""
    c = case(2, 9, 3, 4, 6, 3, 4, seed=29)
    full = run(oracle_mod, c, 4)
    state, ys = c["init"], []
    for t in range(9):
        one = {k: (v[:, t:t + 1] if k in ("x", "dt", "B", "C") else v) for k, v in c.items()}
        one["init"] = state
        o = run(oracle_mod, one, 1)
        ys.append(o["y"])
        state = o["final_state"]
    assert_close(np.concatenate(ys, axis=1), full["y"], 1e-12, "y")
    assert_close(state, full["final_state"], 1e-12, "final")


def test_chunk_states_are_prefix_final_states(oracle_mod):
    c = case(1, 70, 2, 3, 4, 1, 16, seed=17)
    out = run(oracle_mod, c, 16, want_states=True)
    for k in range(out["chunk_states"].shape[2]):
        pre = {kk: (v[:, :16 * k] if kk in ("x", "dt", "B", "C") else v) for kk, v in c.items()}
        ref = run(oracle_mod, pre, 16)["final_state"] if k > 0 else c["init"]
        assert_close(out["chunk_states"][:, :, k], ref, 1e-13, f"chunk {k}")


def test_zero_dt_tokens_leave_state_unchanged(oracle_mod):
    c = case(1, 40, 2, 3, 4, 1, 8, seed=19)
    idx = np.array([3, 4, 17, 30, 39])
    c["dt"][:, idx] = 0.0
    full = run(oracle_mod, c, 8)
    keep = np.setdiff1d(np.arange(40), idx)
    sub = {k: (v[:, keep] if k in ("x", "dt", "B", "C") else v) for k, v in c.items()}
    assert_close(run(oracle_mod, sub, 8)["final_state"], full["final_state"], 1e-13)


@pytest.mark.parametrize("which", ["B", "C"])
def test_zero_B_or_C_gives_skip_only(oracle_mod, which):
    c = case(1, 30, 3, 4, 4, 1, 8, init="zero", seed=23)
    out = run(oracle_mod, c, 8, **{which: np.zeros_like(c[which])})
    assert_close(out["y"], c["D"][None, None, :, None] * c["x"], 1e-15)


def test_single_token_closed_form(oracle_mod):
    c = case(2, 1, 3, 4, 5, 1, 4, init="randn", seed=29)
    out = run(oracle_mod, c, 4)
    for b in range(2):
        for h in range(3):
            dt, x = c["dt"][b, 0, h], c["x"][b, 0, h]
            Bv, Cv = c["B"][b, 0, 0], c["C"][b, 0, 0]
            dec = math.exp(c["A"][h] * dt)
            y = dt * float(Cv @ Bv) * x + dec * (c["init"][b, h] @ Cv) + c["D"][h] * x
            assert_close(out["y"][b, 0, h], y, 1e-14)
            assert_close(out["final_state"][b, h],
                         dec * c["init"][b, h] + dt * np.outer(x, Bv), 1e-14)


def test_linear_in_x_and_init(oracle_mod):
    c1 = case(1, 33, 2, 3, 4, 1, 8, seed=31)
    c2 = case(1, 33, 2, 3, 4, 1, 8, seed=37)
    mix = dict(c1)
    mix["x"] = 2.0 * c1["x"] - 0.5 * c2["x"]
    mix["init"] = 2.0 * c1["init"] - 0.5 * c2["init"]
    c2s = dict(c1)
    c2s["x"], c2s["init"] = c2["x"], c2["init"]
    ya, yb, ym = (run(oracle_mod, cc, 8)["y"] for cc in (c1, c2s, mix))
    assert_close(ym, 2.0 * ya - 0.5 * yb, 1e-12)


def test_identical_heads_in_a_group(oracle_mod):
    """group(h) = h // (H/G): heads 0,1 share group 0, heads 2,3 share group 1."""
    c = case(1, 25, 4, 3, 4, 2, 8, init="zero", seed=41)
    for k in ("x", "dt"):
        c[k][:, :, 1] = c[k][:, :, 0]
        c[k][:, :, 3] = c[k][:, :, 0]
    for k in ("A", "D"):
        c[k][1] = c[k][0]
        c[k][3] = c[k][0]
    y = run(oracle_mod, c, 8)["y"]
    assert np.array_equal(y[:, :, 0], y[:, :, 1])
    # heads 0 and 3 see different B/C groups, so they differ
    assert not np.allclose(y[:, :, 0], y[:, :, 3])


def test_empty_sequence(oracle_mod):
    c = case(1, 4, 2, 3, 4, 1, 8, seed=43)
    e = {k: (v[:, :0] if k in ("x", "dt", "B", "C") else v) for k, v in c.items()}
    out = run(oracle_mod, e, 8, want_states=True)
    assert out["y"].shape == (1, 0, 2, 3)
    assert out["chunk_states"].shape == (1, 2, 0, 3, 4)
    assert_close(out["final_state"], c["init"], 0.0)


def test_bf16_inputs_widen_exactly(oracle_mod):
    """The oracle sees bf16 values widened exactly (no second rounding)."""
    inp = make_inputs(Shape(1, 8, 1, 2, 2, 1, 4), dtype=torch.bfloat16, seed=3)
    xb = inp["x"]
    assert np.array_equal(oracle_mod._f64(xb), xb.float().double().numpy())
