"""Seeded synthetic inputs for the SSD forward.

This module is shared by the tests, the benchmark and the oracle's callers.
It holds only random draws and the input recipe; none of the SSD method's
arithmetic lives here.

Recipe (the Mamba-2 layer's usual input statistics; the source pages,
"Accelerating Mamba-2 forward-pass kernels with CUDA Tile (cuTile)",
section "Mamba-2 前向传播性能基准测试", use bf16 x/B/C with an fp32 state but
print no distributions):

* x ~ N(0, 1)                                  [B, L, H, P]
* dt = softplus(n + bias), n ~ N(0, 0.5^2)     [B, L, H]
  bias[h] = inv_softplus(u), log u ~ U[ln 1e-3, ln 1e-1]   (per head)
* A[h] = -exp(U[0, ln 16])                     (per head, so A in [-16, -1])
* B, C ~ N(0, 1) / sqrt(S)                     [B, L, G, S]
* D[h] ~ N(1, 0.1^2)                           (per head)
* init ~ N(0, 0.1^2) fp32 when requested, else absent (zero state)

Draw order: x, dt noise, bias, A, B, C, D, init.  Draws use numpy's PCG64
generator (identical on x86 and Arm hosts) in float32, then x, B and C are
rounded to the requested dtype (bf16 rounds to nearest even).  dt, A, D and
init stay float32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Shape:
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk_size: int

    @property
    def nchunks(self) -> int:
        return (self.seqlen + self.chunk_size - 1) // self.chunk_size

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen


def _softplus(v: np.ndarray) -> np.ndarray:
    return np.logaddexp(np.float32(0), v).astype(np.float32)


def make_inputs(shape: Shape, dtype: torch.dtype = torch.bfloat16, init: str = "zero",
                seed: int = 0, init_std: float = 0.1) -> dict:
    """Return CPU torch tensors x, dt, A, B, C, D and init (or None).

    ``init`` is "zero" (no initial state) or "randn" (N(0, init_std^2))."""
    if init not in ("zero", "randn"):
        raise ValueError("init must be 'zero' or 'randn'")
    s = shape
    rng = np.random.Generator(np.random.PCG64(seed))
    f32 = np.float32
    x = rng.standard_normal((s.batch, s.seqlen, s.nheads, s.headdim), dtype=f32)
    noise = rng.standard_normal((s.batch, s.seqlen, s.nheads), dtype=f32) * f32(0.5)
    u = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), size=s.nheads)).astype(np.float64)
    bias = np.log(np.expm1(u)).astype(f32)  # inverse softplus, per head
    dt = _softplus(noise + bias[None, None, :])
    A = (-np.exp(rng.uniform(0.0, math.log(16.0), size=s.nheads))).astype(f32)
    scale = f32(1.0 / math.sqrt(s.dstate))
    Bm = rng.standard_normal((s.batch, s.seqlen, s.ngroups, s.dstate), dtype=f32) * scale
    Cm = rng.standard_normal((s.batch, s.seqlen, s.ngroups, s.dstate), dtype=f32) * scale
    D = (1.0 + 0.1 * rng.standard_normal(s.nheads)).astype(f32)
    h0 = None
    if init == "randn":
        h0 = (rng.standard_normal((s.batch, s.nheads, s.headdim, s.dstate), dtype=f32)
              * f32(init_std))

    def t(a, dt_=torch.float32):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dt_)

    return {
        "x": t(x, dtype), "dt": t(dt), "A": t(A), "B": t(Bm, dtype), "C": t(Cm, dtype),
        "D": t(D), "init": None if h0 is None else t(h0),
    }


# Workloads named by what they are (sizes and chunk size).
TINY_FP32 = Shape(batch=1, seqlen=256, nheads=2, headdim=16, dstate=16, ngroups=1, chunk_size=64)
LAYER_2P7B = Shape(batch=4, seqlen=4096, nheads=80, headdim=64, dstate=128, ngroups=1,
                   chunk_size=256)
LONG_S256_G8 = Shape(batch=2, seqlen=32768, nheads=64, headdim=64, dstate=256, ngroups=8,
                     chunk_size=256)
EXTREME_256K = Shape(batch=1, seqlen=262144, nheads=32, headdim=64, dstate=512, ngroups=1,
                     chunk_size=128)
PAGES_EXAMPLE = Shape(batch=4, seqlen=16384, nheads=8, headdim=64, dstate=128, ngroups=1,
                      chunk_size=128)


def sweep_shape(seqlen: int, dstate: int, chunk_size: int, total_tokens: int = 262144) -> Shape:
    """One point of the 1K-256K x dstate sweep: batch*seqlen fixed, 64 heads, P=64, G=1."""
    return Shape(batch=max(1, total_tokens // seqlen), seqlen=seqlen, nheads=64, headdim=64,
                 dstate=dstate, ngroups=1, chunk_size=chunk_size)
