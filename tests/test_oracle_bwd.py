"""Pins of the oracle's backward (CPU only).

``oracle.bwd`` computes the gradients of the token recurrence by its adjoint
recurrence.  The pages name the backward pass without giving it, so it is
pinned to the mathematics:

* central finite differences of the float64 forward (``oracle.fwd``), for
  every element of every input of a small problem with grouped B / C, an
  initial state and a loss that reads both y and the final state;
* the decay-free special case (A = 0, dt = 1), where the forward is causal
  linear attention Y = ((C B^T) * M) X + D X and its gradients have closed
  forms written here with numpy;
* mutants: plausible mistakes planted in a private copy of the C source
  must each fail one of the pins above.
"""
import numpy as np
import pytest
import torch

from state_space_sequence_cumsum_gb300.inputs import Shape, make_inputs


def _f64(t):
    return None if t is None else t.to(torch.float64).numpy()


def small_case(seed=3):
    inp = make_inputs(Shape(2, 7, 4, 3, 5, 2, 4), dtype=torch.float32, init="randn", seed=seed,
                      init_std=0.5)
    c = {k: _f64(v) for k, v in inp.items()}
    rng = np.random.default_rng(seed + 100)
    wy = rng.standard_normal(c["x"].shape)
    wf = rng.standard_normal(c["init"].shape)
    return c, wy, wf


def loss(o, c, wy, wf):
    out = o.fwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], 4, init=c["init"])
    return float(np.sum(out["y"] * wy) + np.sum(out["final_state"] * wf))


GRADS = {"x": "dx", "dt": "ddt", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "init": "dinit"}


def finite_difference_check(o, rtol=1e-6):
    c, wy, wf = small_case()
    g = o.bwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], wy, init=c["init"], dfinal=wf)
    for name, gname in GRADS.items():
        base = c[name]
        fd = np.empty_like(base)
        flat = base.reshape(-1)
        for k in range(flat.size):
            v = flat[k]
            eps = 1e-6 * max(1.0, abs(v))
            flat[k] = v + eps
            up = loss(o, c, wy, wf)
            flat[k] = v - eps
            dn = loss(o, c, wy, wf)
            flat[k] = v
            fd.reshape(-1)[k] = (up - dn) / (2 * eps)
        err = np.max(np.abs(g[gname] - fd))
        scale = max(1.0, float(np.max(np.abs(fd))))
        assert err <= rtol * scale, f"{gname}: max|adjoint - finite difference| = {err:.3e}"


def linear_attention_check(o):
    """A = 0 and dt = 1: Y = ((C B^T) * M) X + D X per (b, h)."""
    inp = make_inputs(Shape(2, 9, 2, 4, 3, 1, 4), dtype=torch.float32, seed=21)
    c = {k: _f64(v) for k, v in inp.items()}
    c["A"] = np.zeros_like(c["A"])
    c["dt"] = np.ones_like(c["dt"])
    rng = np.random.default_rng(5)
    dy = rng.standard_normal(c["x"].shape)
    g = o.bwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], dy)
    L = c["x"].shape[1]
    M = np.tril(np.ones((L, L)))
    dB = np.zeros_like(c["B"])
    dC = np.zeros_like(c["C"])
    for b in range(2):
        Bm, Cm = c["B"][b, :, 0], c["C"][b, :, 0]
        for h in range(2):
            X, dY = c["x"][b, :, h], dy[b, :, h]
            K = (Cm @ Bm.T) * M
            dX = K.T @ dY + c["D"][h] * dY
            assert np.allclose(g["dx"][b, :, h], dX, atol=1e-12), "dx"
            R = (dY @ X.T) * M
            dC[b, :, 0] += R @ Bm
            dB[b, :, 0] += R.T @ Cm
            # with no decay the initial state reaches every output: y_t += h0 C_t
            assert np.allclose(g["dinit"][b, h], dY.T @ Cm, atol=1e-12), "dinit"
    assert np.allclose(g["dB"], dB, atol=1e-12), "dB"
    assert np.allclose(g["dC"], dC, atol=1e-12), "dC"
    dD = np.einsum("blhp,blhp->h", dy, c["x"])
    assert np.allclose(g["dD"], dD, atol=1e-12), "dD"


def test_backward_matches_finite_differences(oracle_mod):
    finite_difference_check(oracle_mod)


def test_backward_decay_free_closed_form(oracle_mod):
    linear_attention_check(oracle_mod)


def test_backward_without_final_state_gradient(oracle_mod):
    """dfinal = None is the same as a zero dfinal."""
    c, wy, _ = small_case(seed=8)
    a = oracle_mod.bwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], wy, init=c["init"])
    b = oracle_mod.bwd(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"], wy, init=c["init"],
                       dfinal=np.zeros_like(c["init"]))
    for k in a:
        assert np.array_equal(a[k], b[k]), k


# (name, text in ssd_oracle.c, replacement): each inside ssd_oracle_bwd
MUTANTS = [
    ("ddt_without_decay_term", "ddt[(b * L + t) * H + h] = ddirect + A[h] * a * da;",
     "ddt[(b * L + t) * H + h] = ddirect;"),
    ("dA_without_dt", "sA += dtv * a * da;", "sA += a * da;"),
    ("adjoint_not_decayed", "adj[k] *= a;", "adj[k] *= 1.0;"),
    ("dC_from_previous_state", "acc += ht[p * S + s] * dyt[p];", "acc += hprev[p * S + s] * dyt[p];"),
    ("dx_without_skip", "dxt[p] = D[h] * dyt[p] + dtv * hb;", "dxt[p] = dtv * hb;"),
    ("dB_without_dt", "dbt[s] += dtv * acc;", "dbt[s] += acc;"),
    ("da_with_current_state", "da += adj[p * S + s] * hprev[p * S + s];",
     "da += adj[p * S + s] * ht[p * S + s];"),
    ("dB_transposed_state", "acc += adj[p * S + s] * xt[p];", "acc += adj[s * P + p % S] * xt[p];"),
]


def _bwd_battery(o):
    failed = []
    for name, fn in (("finite_differences", lambda: finite_difference_check(o)),
                     ("linear_attention", lambda: linear_attention_check(o))):
        try:
            fn()
        except (AssertionError, ValueError, IndexError):
            failed.append(name)
    return failed


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_backward_mutant_is_caught(oracle_mod, tmp_path, name, old, new):
    src = oracle_mod.source_text()
    start = src.index("int ssd_oracle_bwd(")
    assert old in src[start:], f"mutation site for {name} not found"
    mutated = src[:start] + src[start:].replace(old, new, 1)
    so = oracle_mod.compile_source(mutated, str(tmp_path / f"mut_{name}.so"))
    assert _bwd_battery(oracle_mod.Variant(so)), f"mutant {name} passed every pin"
