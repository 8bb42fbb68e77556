"""Shared helpers for the GPU parity tests: run the CUDA path and the oracle on
the same seeded inputs and compare element by element.

Tolerances (written here, used by every parity test): the output and the
states must satisfy max|gpu - oracle| <= tol * rms(oracle) with
tol = 2e-2 for bf16 inputs (bf16 MMA operands, f32 accumulation) and
tol = 1e-4 for f32 inputs (f32 arithmetic throughout).
"""
import numpy as np
import torch

import oracle
from state_space_sequence_cumsum_gb300.inputs import Shape, make_inputs

TOL = {torch.bfloat16: 2e-2, torch.float32: 1e-4}


def to_gpu(inp):
    return {k: (None if v is None else v.cuda()) for k, v in inp.items()}


def rel_err(gpu, ref):
    """max|gpu - ref| / rms(ref) (rms floored at 1e-30 for all-zero refs)."""
    g = gpu.detach().to("cpu", torch.float64).numpy() if hasattr(gpu, "detach") else gpu
    if ref.size == 0:
        return 0.0
    rms = max(float(np.sqrt(np.mean(ref * ref))), 1e-30)
    return float(np.max(np.abs(g - ref))) / rms


def assert_parity(gpu, ref, dtype, what):
    assert tuple(gpu.shape) == tuple(ref.shape), f"{what}: shape {tuple(gpu.shape)} vs {ref.shape}"
    g = gpu.detach().to("cpu", torch.float64).numpy()
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    e = rel_err(g, ref)
    assert e <= TOL[dtype], f"{what}: max|err|/rms = {e:.3e} > {TOL[dtype]:.0e}"
    return e


def oracle_run(inp, T, want_states=False, heads=None):
    """Oracle on (optionally) a subset of heads; inputs are the CPU tensors."""
    x, dt, A, Bm, Cm, D, init = (inp[k] for k in ("x", "dt", "A", "B", "C", "D", "init"))
    if heads is not None:
        H, G = x.shape[2], Bm.shape[2]
        hpg = H // G
        heads = list(heads)
        groups = sorted({h // hpg for h in heads})
        # keep whole groups so group(h) stays consistent: take every head of the groups
        heads = [h for g in groups for h in range(g * hpg, (g + 1) * hpg)]
        idx = torch.tensor(heads)
        gidx = torch.tensor(groups)
        x, dt, A, D = x[:, :, idx], dt[:, :, idx], A[idx], D[idx]
        Bm, Cm = Bm[:, :, gidx], Cm[:, :, gidx]
        init = None if init is None else init[:, idx]
    out = oracle.fwd(x, dt, A, Bm, Cm, D, T, init=init, want_states=want_states)
    out["heads"] = heads
    return out


def case_inputs(B, L, H, P, S, G, T, dtype=torch.bfloat16, init="zero", seed=0):
    return make_inputs(Shape(B, L, H, P, S, G, T), dtype=dtype, init=init, seed=seed)
