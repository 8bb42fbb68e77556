"""Float64 CPU oracle for the Mamba-2 chunked SSD forward.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline / reference leg may import this package.
The product library (``state_space_sequence_cumsum_gb300``) never imports
it and shares no code with it; the two meet only through the seeded input
generator, which contains none of the method's arithmetic.

What it computes follows "Accelerating Mamba-2 forward-pass kernels with
CUDA Tile (cuTile)" (dbyun.net/article/14364):

* ``fwd``           -- section "Mamba-2 架构", the token recurrence
  h_t = exp(A dt_t) h_{t-1} + dt_t B_t x_t^T, y_t = C_t^T h_t + D x_t, plus
  every chunk's start state and the final state as section
  "Kernel 2: fwd_pass_state" defines them.
* ``chunk_cumsum``  -- section "Kernel 1": the within-chunk cumulative sum of
  A[h]*dt scaled by log2(e).
* ``gated_rmsnorm`` -- the gate and RMS normalisation that follow the scan
  (the post's operator-fusion section names them; the Mamba-2 form, y times
  silu(z) then a grouped RMS norm and a per-channel weight, is the reading).
* ``bwd``           -- the gradients of ``fwd``'s recurrence with respect to
  every input, by the adjoint recurrence (reverse-mode differentiation of
  the same token loop; the pages name the backward pass but do not give
  it).  Pinned by central finite differences.

The arithmetic lives in ``ssd_oracle.c`` (plain C, float64, OpenMP over
(batch, head)).  Inputs of any dtype are widened exactly to float64 before
the call.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``ssd_oracle.c`` into ``liboracle.so`` with gcc (-O2, OpenMP).

    No fast-math: the oracle keeps IEEE float64 semantics."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11",
           "-Wall", "-Wextra", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    i64, dp = ctypes.c_int64, ctypes.POINTER(ctypes.c_double)
    lib.ssd_oracle_chunk_cumsum.argtypes = [i64, i64, i64, i64, dp, dp, dp]
    lib.ssd_oracle_chunk_cumsum.restype = ctypes.c_int
    lib.ssd_oracle_fwd.argtypes = [i64] * 7 + [dp] * 10 + [ctypes.c_int]
    lib.ssd_oracle_fwd.restype = ctypes.c_int
    lib.ssd_oracle_bwd.argtypes = [i64] * 6 + [dp] * 16 + [ctypes.c_int]
    lib.ssd_oracle_bwd.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB_PATH)
    return _lib


def _f64(a) -> np.ndarray:
    """Exact widening of a torch tensor or array to contiguous float64."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor (bf16 has no numpy dtype)
        import torch
        a = a.detach().to("cpu", torch.float64).contiguous().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def chunk_cumsum(dt, A, chunk_size: int, _lib_override=None) -> np.ndarray:
    """G[b, h, t] = log2(e) * sum_{t'=c*T}^{t} A[h] * dt[b, t', h], c = t // T.

    Returns float64 [B, H, L] (token-contiguous, the layout the pages move
    decay_cumsum to in "Mamba-2 性能优化")."""
    dt, A = _f64(dt), _f64(A)
    B, L, H = dt.shape
    G = np.empty((B, H, L), dtype=np.float64)
    rc = (_lib_override or _load()).ssd_oracle_chunk_cumsum(B, L, H, int(chunk_size), _ptr(dt), _ptr(A), _ptr(G))
    if rc != 0:
        raise ValueError(f"oracle chunk_cumsum rejected its arguments (rc={rc})")
    return G


def fwd(x, dt, A, Bm, Cm, D, chunk_size: int, init=None, want_states: bool = False,
        nthreads: int = 0, _lib_override=None) -> dict:
    """Run the float64 token recurrence.

    Shapes: x [B,L,H,P], dt [B,L,H], A [H], Bm/Cm [B,L,G,S], D [H],
    init [B,H,P,S] or None (zeros).  Returns a dict with ``y`` [B,L,H,P],
    ``final_state`` [B,H,P,S] and, if ``want_states``, ``chunk_states``
    [B,H,nc,P,S] where chunk_states[:, :, c] is the state before token
    c*chunk_size."""
    x, dt, A, Bm, Cm, D, init = (_f64(v) for v in (x, dt, A, Bm, Cm, D, init))
    B, L, H, P = x.shape
    G, S = Bm.shape[2], Bm.shape[3]
    T = int(chunk_size)
    nc = (L + T - 1) // T
    if dt.shape != (B, L, H) or Bm.shape != (B, L, G, S) or Cm.shape != (B, L, G, S):
        raise ValueError("oracle fwd: inconsistent input shapes")
    if A.shape != (H,) or D.shape != (H,):
        raise ValueError("oracle fwd: A and D must be [H]")
    if init is not None and init.shape != (B, H, P, S):
        raise ValueError("oracle fwd: init must be [B,H,P,S]")
    y = np.empty((B, L, H, P), dtype=np.float64)
    final = np.empty((B, H, P, S), dtype=np.float64)
    states = np.empty((B, H, nc, P, S), dtype=np.float64) if want_states else None
    rc = (_lib_override or _load()).ssd_oracle_fwd(
        B, L, H, P, S, G, T, _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(D),
        _ptr(init), _ptr(y), _ptr(final), _ptr(states), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle fwd failed (rc={rc})")
    out = {"y": y, "final_state": final}
    if want_states:
        out["chunk_states"] = states
    return out


def bwd(x, dt, A, Bm, Cm, D, dy, init=None, dfinal=None, nthreads: int = 0,
        _lib_override=None) -> dict:
    """Gradients of the token recurrence by its adjoint (float64).

    For a scalar loss with dloss/dy = dy [B,L,H,P] and dloss/dfinal = dfinal
    [B,H,P,S] (None: zero), returns dx, ddt, dA, dB, dC, dD and dinit
    (dinit is the gradient with respect to the initial state, zeros when
    init is None)."""
    x, dt, A, Bm, Cm, D, dy, init, dfinal = (_f64(v) for v in (x, dt, A, Bm, Cm, D, dy, init,
                                                                 dfinal))
    B, L, H, P = x.shape
    G, S = Bm.shape[2], Bm.shape[3]
    if dy.shape != x.shape or dt.shape != (B, L, H) or Bm.shape != (B, L, G, S) \
            or Cm.shape != Bm.shape or A.shape != (H,) or D.shape != (H,):
        raise ValueError("oracle bwd: inconsistent input shapes")
    for st in (init, dfinal):
        if st is not None and st.shape != (B, H, P, S):
            raise ValueError("oracle bwd: states must be [B,H,P,S]")
    out = {"dx": np.empty_like(x), "ddt": np.empty_like(dt), "dA": np.empty(H),
           "dB": np.empty_like(Bm), "dC": np.empty_like(Cm), "dD": np.empty(H),
           "dinit": np.empty((B, H, P, S))}
    rc = (_lib_override or _load()).ssd_oracle_bwd(
        B, L, H, P, S, G, _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(D), _ptr(init),
        _ptr(dy), _ptr(dfinal), _ptr(out["dx"]), _ptr(out["ddt"]), _ptr(out["dA"]),
        _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]), _ptr(out["dinit"]), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle bwd failed (rc={rc})")
    return out


def gated_rmsnorm(y, z, weight, eps: float, group_size: int) -> np.ndarray:
    """The output epilogue that follows the scan ("Mamba-2 forward-pass
    kernels" post, section on operator fusion: gating and normalisation after
    the scan), in its Mamba-2 form: per token, with g = y * silu(z) and
    silu(z) = z / (1 + exp(-z)),
        out = g / sqrt(mean(g^2 over each group of group_size channels) + eps) * weight.
    y, z: [..., D] (D = nheads * headdim channels per token, any dtype, widened
    exactly); weight [D]; returns float64 [..., D]."""
    y, z, w = _f64(y), _f64(z), _f64(weight)
    D = y.shape[-1]
    if z.shape != y.shape or w.shape != (D,) or group_size <= 0 or D % group_size:
        raise ValueError("oracle gated_rmsnorm: inconsistent shapes")
    g = y * (z / (1.0 + np.exp(-z)))
    gg = g.reshape(g.shape[:-1] + (D // group_size, group_size))
    ms = np.mean(gg * gg, axis=-1, keepdims=True)
    return (gg / np.sqrt(ms + eps)).reshape(g.shape) * w


def cpu_cores() -> int:
    """Threads the oracle's OpenMP loop uses by default on this host."""
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


class Variant:
    """The oracle's Python entry points bound to another build of the C source.

    Used only by the mutation tests, which compile deliberately broken copies
    of ``ssd_oracle.c`` to show that the pins detect plausible mistakes."""

    def __init__(self, so_path: str):
        self._lib = _bind(so_path)

    def fwd(self, *args, **kw):
        return fwd(*args, _lib_override=self._lib, **kw)

    def chunk_cumsum(self, *args, **kw):
        return chunk_cumsum(*args, _lib_override=self._lib, **kw)

    def bwd(self, *args, **kw):
        return bwd(*args, _lib_override=self._lib, **kw)

    _f64 = staticmethod(_f64)


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def compile_source(text: str, out_path: str) -> str:
    """Compile C source text with the oracle's flags (mutation tests only)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(text)
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", src, "-o",
                    out_path, "-lm"], check=True)
    return out_path
