"""Tensor-level binding of the C ABI (same names as ``include/ssd.h``).

PyTorch only allocates outputs/workspace and supplies the current CUDA
stream; every arithmetic step runs in the library's kernels.  Inputs must be
contiguous CUDA tensors on one device: x, B, C in bf16 or f32 (one dtype),
dt, A, D and states in f32.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import SsdError, check, dims as _dims

__all__ = ["ssd_chunk_cumsum", "ssd_state_pass", "ssd_chunk_out", "ssd_state_out", "ssd_fwd",
           "ssd_fwd_path", "ssd_fwd_plan", "ssd_fwd_staged",
           "ssd_fwd_workspace_size", "ssd_fwd_chosen_chunk_size", "ssd_fwd_chunk_size_was_timed",
           "ssd_stream_status",
           "ssd_fwd_host", "ssd_segment_summary", "ssd_carry_in", "ssd_fwd_context_parallel",
           "ssd_status_string", "ssd_decode_step", "ssd_bwd", "ssd_gated_rmsnorm",
           "SsdFunction", "SsdError",
           "Workspace"]


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return _lib.SSD_BF16
    if t.dtype == torch.float32:
        return _lib.SSD_F32
    raise TypeError(f"x/B/C must be bfloat16 or float32, got {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("SSD tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("SSD tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else None


def _f32(t, name):
    if t is not None and t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    return t


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _geom(x, B):
    b, L, H, P = x.shape
    if B.dim() != 4 or B.shape[0] != b or B.shape[1] != L:
        raise ValueError("B/C must be [batch, seqlen, ngroups, dstate]")
    return _dims(b, L, H, P, B.shape[3], B.shape[2])


def ssd_status_string(status: int) -> str:
    return _lib.status_string(status)


def ssd_chunk_cumsum(dt, A, chunk_size, G_cum=None, dt_t=None, want_dt_t=True, stream=None):
    """Stage 1.  Returns (G_cum [B,H,L] f32, dt_t [B,H,L] f32 or None)."""
    _f32(dt, "dt"), _f32(A, "A")
    b, L, H = dt.shape
    if G_cum is None:
        G_cum = torch.empty((b, H, L), device=dt.device, dtype=torch.float32)
    if dt_t is None and want_dt_t:
        dt_t = torch.empty((b, H, L), device=dt.device, dtype=torch.float32)
    d = _dims(b, L, H, 1, 1, 1)
    check(_lib.load().ssd_chunk_cumsum(_ptr(dt), _ptr(A), _ptr(G_cum), _ptr(dt_t), d,
                                       int(chunk_size), _stream(stream)), "ssd_chunk_cumsum")
    return G_cum, dt_t


def ssd_state_pass(x, B, dt_t, G_cum, chunk_size, init_state=None, chunk_states=True,
                   final_state=True, stream=None):
    """Stage 2.  chunk_states / final_state: True = allocate, None/False = skip,
    or a preallocated f32 tensor.  Returns (chunk_states, final_state)."""
    d = _geom(x, B)
    nc = (d.seqlen + chunk_size - 1) // chunk_size
    dev = x.device
    if chunk_states is True:
        chunk_states = torch.empty((d.batch, d.nheads, nc, d.headdim, d.dstate), device=dev,
                                   dtype=torch.float32)
    if final_state is True:
        final_state = torch.empty((d.batch, d.nheads, d.headdim, d.dstate), device=dev,
                                  dtype=torch.float32)
    chunk_states = chunk_states if isinstance(chunk_states, torch.Tensor) else None
    final_state = final_state if isinstance(final_state, torch.Tensor) else None
    _f32(init_state, "init_state")
    check(_lib.load().ssd_state_pass(_ptr(x), _ptr(B), _ptr(dt_t), _ptr(G_cum),
                                     _ptr(init_state), _ptr(chunk_states), _ptr(final_state), d,
                                     _dtype_code(x), int(chunk_size), _stream(stream)),
          "ssd_state_pass")
    return chunk_states, final_state


def ssd_chunk_out(x, B, C, dt_t, G_cum, chunk_states, D, chunk_size, y=None, stream=None):
    """Stage 3.  Returns y [B,L,H,P] in x's dtype."""
    d = _geom(x, B)
    if y is None:
        y = torch.empty_like(x)
    check(_lib.load().ssd_chunk_out(_ptr(x), _ptr(B), _ptr(C), _ptr(dt_t), _ptr(G_cum),
                                    _ptr(chunk_states), _ptr(_f32(D, "D")), _ptr(y), d,
                                    _dtype_code(x), int(chunk_size), _stream(stream)),
          "ssd_chunk_out")
    return y


def ssd_decode_step(x, dt, A, B, C, D, state, state_out=None, y=None, stream=None):
    """One token of the recurrence on a carried state.

    x [batch, 1, H, P] (or [batch, H, P]), dt [batch, 1, H] (or [batch, H]),
    B, C [batch, 1, G, S] (or [batch, G, S]) in x's dtype; A, D [H] f32;
    state [batch, H, P, S] f32.  The updated state goes to ``state_out``
    (default: ``state`` itself, updated in place).  Returns (y, state_out),
    y shaped like x."""
    x4 = x if x.dim() == 4 else x.unsqueeze(1)
    B4 = B if B.dim() == 4 else B.unsqueeze(1)
    C4 = C if C.dim() == 4 else C.unsqueeze(1)
    d = _geom(x4, B4)
    if C4.shape != B4.shape:
        raise ValueError("B and C must have the same shape")
    if d.seqlen != 1:
        raise ValueError("the decode step takes one token")
    if tuple(state.shape) != (d.batch, d.nheads, d.headdim, d.dstate):
        raise ValueError("state must be [batch, nheads, headdim, dstate]")
    if state_out is None:
        state_out = state
    if y is None:
        y = torch.empty_like(x)
    check(_lib.load().ssd_decode_step(_ptr(x), _ptr(_f32(dt, "dt")), _ptr(_f32(A, "A")), _ptr(B),
                                      _ptr(C), _ptr(_f32(D, "D")), _ptr(_f32(state, "state")),
                                      _ptr(_f32(state_out, "state_out")), _ptr(y), d,
                                      _dtype_code(x), _stream(stream)),
          "ssd_decode_step")
    return y, state_out


def ssd_gated_rmsnorm(y, z, weight, eps=1e-5, group_size=None, out=None, stream=None):
    """out = rmsnorm(y * silu(z)) * weight over groups of ``group_size``
    channels of the last dimension (default: all of it); y and z of one
    dtype (bf16 or f32) and shape [..., dim], weight [dim] f32.  ``out`` may
    be y or z (in place)."""
    if z.shape != y.shape or z.dtype != y.dtype:
        raise ValueError("y and z must have the same shape and dtype")
    dim = y.shape[-1]
    gs = dim if group_size is None else int(group_size)
    if out is None:
        out = torch.empty_like(y)
    check(_lib.load().ssd_gated_rmsnorm(_ptr(y), _ptr(z), _ptr(_f32(weight, "weight")), _ptr(out),
                                        y.numel() // dim if dim else 0, dim, gs, float(eps),
                                        _dtype_code(y), _stream(stream)),
          "ssd_gated_rmsnorm")
    return out


def ssd_bwd(x, dt, A, B, C, D, dy, initial_state=None, dfinal=None, want_dinit=True,
            workspace=None, stream=None):
    """Gradients of ssd_fwd's outputs (y and the final state) with respect to
    every input.  dy is the loss gradient of y (x's dtype), dfinal that of
    the final state (f32, None = zero).  Returns a dict with dx, ddt, dA, dB,
    dC, dD and dinit (None unless want_dinit)."""
    d = _geom(x, B)
    code = _dtype_code(x)
    lib = _lib.load()
    nbytes = lib.ssd_bwd_workspace_size(d, code)
    if nbytes == 0:
        raise ValueError("ssd_bwd: invalid sizes")
    ws = workspace if workspace is not None else Workspace()
    buf = ws.get(nbytes, x.device)
    out = {"dx": torch.empty_like(x), "ddt": torch.empty_like(dt),
           "dA": torch.empty_like(A), "dB": torch.empty_like(B), "dC": torch.empty_like(C),
           "dD": torch.empty_like(D),
           "dinit": (torch.empty((d.batch, d.nheads, d.headdim, d.dstate), dtype=torch.float32,
                                 device=x.device) if want_dinit else None)}
    check(lib.ssd_bwd(_ptr(x), _ptr(_f32(dt, "dt")), _ptr(_f32(A, "A")), _ptr(B), _ptr(C),
                      _ptr(_f32(D, "D")), _ptr(_f32(initial_state, "initial_state")), _ptr(dy),
                      _ptr(_f32(dfinal, "dfinal")), _ptr(out["dx"]), _ptr(out["ddt"]),
                      _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]),
                      _ptr(out["dinit"]), d, code, ctypes.c_void_p(buf.data_ptr()),
                      ctypes.c_size_t(nbytes), _stream(stream)),
          "ssd_bwd")
    return out


class SsdFunction(torch.autograd.Function):
    """torch.autograd binding: forward is ssd_fwd (y, final state), backward
    is ssd_bwd.  Both run in the library's kernels."""

    @staticmethod
    def forward(ctx, x, dt, A, B, C, D, initial_state=None):
        y, final, _ = ssd_fwd(x, dt, A, B, C, D, chunk_size=0, initial_state=initial_state,
                              return_final_state=True)
        ctx.save_for_backward(x, dt, A, B, C, D, initial_state)
        return y, final

    @staticmethod
    def backward(ctx, dy, dfinal):
        x, dt, A, B, C, D, init = ctx.saved_tensors
        g = ssd_bwd(x, dt, A, B, C, D, dy.contiguous(), initial_state=init,
                    dfinal=None if dfinal is None else dfinal.contiguous(),
                    want_dinit=init is not None)
        return g["dx"], g["ddt"], g["dA"], g["dB"], g["dC"], g["dD"], g["dinit"]


def ssd_fwd_workspace_size(batch, seqlen, nheads, headdim, dstate, ngroups, dtype, chunk_size,
                           want_chunk_states) -> int:
    code = _lib.SSD_BF16 if dtype == torch.bfloat16 else _lib.SSD_F32
    return int(_lib.load().ssd_fwd_workspace_size(
        _dims(batch, seqlen, nheads, headdim, dstate, ngroups), code, int(chunk_size),
        int(bool(want_chunk_states))))


def ssd_fwd_chosen_chunk_size(batch, seqlen, nheads, headdim, dstate, ngroups, dtype) -> int:
    """The chunk size ssd_fwd(chunk_size=0) uses for this shape; fixes the
    choice if no call has fixed it yet (see include/ssd.h)."""
    code = _lib.SSD_BF16 if dtype == torch.bfloat16 else _lib.SSD_F32
    return int(_lib.load().ssd_fwd_chosen_chunk_size(
        _dims(batch, seqlen, nheads, headdim, dstate, ngroups), code))


def ssd_fwd_chunk_size_was_timed(batch, seqlen, nheads, headdim, dstate, ngroups, dtype) -> bool:
    """True if this shape's chunk size was fixed by timing the candidates."""
    code = _lib.SSD_BF16 if dtype == torch.bfloat16 else _lib.SSD_F32
    return bool(_lib.load().ssd_fwd_chunk_size_was_timed(
        _dims(batch, seqlen, nheads, headdim, dstate, ngroups), code))


class Workspace:
    """Reusable device workspace for ssd_fwd (grown on demand, 256-byte aligned)
    plus named buffers for the stage-by-stage form of the same pass."""

    def __init__(self, device=None):
        self.device = device
        self.buf = None
        self.named = {}

    def get(self, nbytes: int, device) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes or self.buf.device != device:
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        return self.buf

    def tensor(self, name, shape, dtype, device) -> torch.Tensor:
        t = self.named.get(name)
        if t is None or tuple(t.shape) != tuple(shape) or t.dtype != dtype or t.device != device:
            t = torch.empty(shape, dtype=dtype, device=device)
            self.named[name] = t
        return t


def ssd_fwd(x, dt, A, B, C, D, chunk_size=0, initial_state=None, return_final_state=True,
            return_chunk_states=False, y=None, final_state=None, chunk_states=None,
            workspace: Workspace | None = None, stream=None):
    """Whole SSD forward.  Returns (y, final_state or None, chunk_states or None)."""
    d = _geom(x, B)
    for t, n in ((dt, "dt"), (A, "A"), (D, "D"), (initial_state, "initial_state")):
        _f32(t, n)
    code = _dtype_code(x)
    lib = _lib.load()
    T = int(chunk_size)
    want_states = chunk_states is not None or return_chunk_states
    if T == 0 and want_states:
        # the chunk states' count depends on the chunk size: fix the choice now
        T = int(lib.ssd_fwd_chosen_chunk_size(d, code))
        if T <= 0:
            raise SsdError(_lib.SSD_ERR_INVALID_ARG, "ssd_fwd")
    dev = x.device
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and return_final_state:
        final_state = torch.empty((d.batch, d.nheads, d.headdim, d.dstate), device=dev,
                                  dtype=torch.float32)
    if chunk_states is None and return_chunk_states:
        nc = (d.seqlen + T - 1) // T
        chunk_states = torch.empty((d.batch, d.nheads, nc, d.headdim, d.dstate), device=dev,
                                   dtype=torch.float32)
    # chunk_size 0 without chunk states: the library chooses (and the first
    # such call for a shape times the candidates on these buffers)
    nbytes = int(lib.ssd_fwd_workspace_size(d, code, T, int(chunk_states is not None)))
    ws = (workspace or Workspace()).get(nbytes, dev)
    check(lib.ssd_fwd(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                      _ptr(initial_state), _ptr(y), _ptr(final_state), _ptr(chunk_states), d,
                      code, T, _ptr(ws), ctypes.c_size_t(ws.numel()), _stream(stream)), "ssd_fwd")
    return y, final_state, chunk_states


def _host_ptr(t):
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError("ssd_fwd_host takes host (CPU) tensors")
    if not t.is_contiguous():
        raise ValueError("SSD tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else None


def ssd_fwd_host(x, dt, A, B, C, D, chunk_size=0, initial_state=None, y=None,
                 final_state=True, workspace: Workspace | None = None, device=None, stream=None):
    """Whole SSD forward from host tensors to host tensors (ssd_fwd_host: the
    copies overlap the kernels).  Inputs and outputs are CPU tensors, pinned
    for asynchronous copies; the call returns before the work ends --
    synchronize `stream` (default: the current stream of `device`) before
    reading y.  Returns (y, final_state or None)."""
    d = _geom(x, B)
    for t, n in ((dt, "dt"), (A, "A"), (D, "D"), (initial_state, "initial_state")):
        _f32(t, n)
    code = _dtype_code(x)
    lib = _lib.load()
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if y is None:
        y = torch.empty(x.shape, dtype=x.dtype).pin_memory()
    if final_state is True:
        final_state = torch.empty((d.batch, d.nheads, d.headdim, d.dstate),
                                  dtype=torch.float32).pin_memory()
    elif final_state is False:
        final_state = None
    nbytes = int(lib.ssd_fwd_host_workspace_size(d, code, int(chunk_size)))
    if nbytes == 0:
        raise SsdError(_lib.SSD_ERR_INVALID_ARG, "ssd_fwd_host")
    ws = (workspace or Workspace()).get(nbytes, dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        check(lib.ssd_fwd_host(_host_ptr(x), _host_ptr(dt), _host_ptr(A), _host_ptr(B),
                               _host_ptr(C), _host_ptr(D), _host_ptr(initial_state), _host_ptr(y),
                               _host_ptr(final_state), d, code, int(chunk_size), _ptr(ws),
                               ctypes.c_size_t(ws.numel()), ctypes.c_void_p(s.cuda_stream)),
              "ssd_fwd_host")
    return y, final_state


def ssd_state_out(x, B, C, dt_t, G_cum, D, chunk_size, initial_state=None, y=None,
                  final_state=True, chunk_states=None, workspace: "Workspace | None" = None,
                  stream=None):
    """Fused stages 2+3 (tensor-core path).  Returns (y, final_state, chunk_states)."""
    d = _geom(x, B)
    nc = (d.seqlen + chunk_size - 1) // chunk_size
    dev = x.device
    if y is None:
        y = torch.empty_like(x)
    if final_state is True:
        final_state = torch.empty((d.batch, d.nheads, d.headdim, d.dstate), device=dev,
                                  dtype=torch.float32)
    if chunk_states is True:
        chunk_states = torch.empty((d.batch, d.nheads, nc, d.headdim, d.dstate), device=dev,
                                   dtype=torch.float32)
    final_state = final_state if isinstance(final_state, torch.Tensor) else None
    chunk_states = chunk_states if isinstance(chunk_states, torch.Tensor) else None
    lib = _lib.load()
    code = _dtype_code(x)
    nbytes = int(lib.ssd_state_out_workspace_size(d, code, int(chunk_size))) or 256
    ws = (workspace or Workspace()).get(nbytes, dev)
    check(lib.ssd_state_out(_ptr(x), _ptr(B), _ptr(C), _ptr(dt_t), _ptr(G_cum),
                            _ptr(_f32(D, "D")), _ptr(_f32(initial_state, "init")), _ptr(y),
                            _ptr(final_state), _ptr(chunk_states), d, code, int(chunk_size),
                            _ptr(ws), ctypes.c_size_t(ws.numel()), _stream(stream)),
          "ssd_state_out")
    return y, final_state, chunk_states


def ssd_fwd_path(x, B, chunk_size=0, want_states=False) -> str:
    """Name of the kernel path ssd_fwd takes for these arguments."""
    d = _geom(x, B)
    code = _lib.load().ssd_fwd_path(d, _dtype_code(x), int(chunk_size), int(bool(want_states)))
    return _lib.PATH_NAMES.get(code, "invalid")


def ssd_fwd_plan(x, B, chunk_size, want_states=False) -> dict:
    """The C-ABI stage calls ssd_fwd makes for these arguments, in order."""
    path = ssd_fwd_path(x, B, chunk_size, want_states)
    if path == "fused-pair-tensor-cores":
        kernels = ["fused_pair"]  # one kernel: ssd_fwd itself
    elif path == "fused-tensor-cores":
        kernels = ["chunk_cumsum", "state_out"]
    else:
        kernels = ["chunk_cumsum", "state_pass", "chunk_out"]
    return {"path": path, "chunk_size": int(chunk_size), "kernels": kernels}


def ssd_fwd_staged(plan, x, dt, A, B, C, D, initial_state, y, final_state, chunk_states,
                   workspace: Workspace, events=None, stream=None):
    """ssd_fwd as its individual stage calls (same kernels, same order), with an
    optional CUDA event recorded before the first and after every stage on the
    launching stream.  Used to time each kernel inside a whole pass."""
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    b, L, H, P = x.shape
    Sd = B.shape[3]
    T = plan["chunk_size"]
    dev = x.device

    def mark(i):
        if events is not None:
            events[i].record(s)

    if plan["kernels"] == ["fused_pair"]:
        mark(0)
        ssd_fwd(x, dt, A, B, C, D, chunk_size=plan.get("call_chunk_size", T),
                initial_state=initial_state, y=y,
                final_state=final_state, chunk_states=chunk_states,
                return_final_state=final_state is not None,
                return_chunk_states=chunk_states is not None, workspace=workspace, stream=s)
        mark(1)
        return y, final_state, chunk_states
    Gc = workspace.tensor("G_cum", (b, H, L), torch.float32, dev)
    dtT = workspace.tensor("dt_t", (b, H, L), torch.float32, dev)
    nc = (L + T - 1) // T
    states = chunk_states
    if states is None and plan["kernels"][1] != "state_out":
        states = workspace.tensor("chunk_states", (b, H, nc, P, Sd), torch.float32, dev)

    mark(0)
    ssd_chunk_cumsum(dt, A, T, G_cum=Gc, dt_t=dtT, stream=s)
    mark(1)
    if plan["kernels"][1] == "state_out":
        ssd_state_out(x, B, C, dtT, Gc, D, T, initial_state=initial_state, y=y,
                      final_state=final_state if final_state is not None else False,
                      chunk_states=chunk_states, workspace=workspace, stream=s)
        mark(2)
        return y, final_state, chunk_states
    ssd_state_pass(x, B, dtT, Gc, T, init_state=initial_state, chunk_states=states,
                   final_state=final_state if final_state is not None else False, stream=s)
    mark(2)
    ssd_chunk_out(x, B, C, dtT, Gc, states, D, T, y=y, stream=s)
    mark(3)
    return y, final_state, chunk_states


def ssd_segment_summary(x, dt, A, B, chunk_size, workspace: "Workspace | None" = None,
                        stream=None):
    """Step 1 of the sequence-sharded forward: this segment's end state from a
    zero state [batch, H, P, S] f32 and its total decay [batch, H] f32 (log2
    units).  Returns (seg_state, seg_decay)."""
    d = _geom(x, B)
    code = _dtype_code(x)
    lib = _lib.load()
    dev = x.device
    seg_state = torch.empty((d.batch, d.nheads, d.headdim, d.dstate), device=dev,
                            dtype=torch.float32)
    seg_decay = torch.empty((d.batch, d.nheads), device=dev, dtype=torch.float32)
    nbytes = int(lib.ssd_segment_summary_workspace_size(d, code, int(chunk_size)))
    if nbytes == 0:
        raise SsdError(_lib.SSD_ERR_INVALID_ARG, "ssd_segment_summary")
    ws = (workspace or Workspace()).get(nbytes, dev)
    check(lib.ssd_segment_summary(_ptr(x), _ptr(_f32(dt, "dt")), _ptr(_f32(A, "A")), _ptr(B),
                                  _ptr(seg_state), _ptr(seg_decay), d, code, int(chunk_size),
                                  _ptr(ws), ctypes.c_size_t(ws.numel()), _stream(stream)),
          "ssd_segment_summary")
    return seg_state, seg_decay


def ssd_carry_in(seg_states, seg_decays, upto, initial_state=None, out=None, stream=None):
    """Step 3 of the sequence-sharded forward: the state carried into segment
    `upto` from the gathered summaries seg_states [R, batch, H, P, S] and
    seg_decays [R, batch, H] (f32, one entry per segment in sequence order)
    and the sequence's initial state (None: zeros).  Returns h_in."""
    R, b, H, P, S = seg_states.shape
    if tuple(seg_decays.shape) != (R, b, H):
        raise ValueError("seg_decays must be [segments, batch, nheads]")
    if out is None:
        out = torch.empty((b, H, P, S), device=seg_states.device, dtype=torch.float32)
    d = _dims(b, 1, H, P, S, 1)
    check(_lib.load().ssd_carry_in(_ptr(_f32(seg_states, "seg_states")),
                                   _ptr(_f32(seg_decays, "seg_decays")),
                                   _ptr(_f32(initial_state, "initial_state")), int(R), int(upto),
                                   _ptr(out), d, _stream(stream)),
          "ssd_carry_in")
    return out


def ssd_fwd_context_parallel(x, dt, A, B, C, D, chunk_size, initial_state=None, group=None,
                             return_chunk_states=False, workspace: "Workspace | None" = None,
                             stream=None):
    """Sequence-sharded forward over the ranks of a torch.distributed group:
    rank r holds the r-th contiguous segment of every sequence (x, dt, B, C
    of its tokens; A, D and the sequence's initial state are the same on
    every rank).  One all-gather of the per-segment summaries, then each rank
    runs its segment from its carried-in state.  Returns this segment's
    (y, final_state, chunk_states or None); the last rank's final state is the
    sequence's.  With chunk states, every segment but the last must be a
    whole number of chunks for them to line up with the unsharded run's."""
    import torch.distributed as dist
    R = dist.get_world_size(group)
    r = dist.get_rank(group)
    b, _, H, P = x.shape
    Sd = B.shape[3]
    n_state = b * H * P * Sd
    if r < R - 1:
        s_r, d_r = ssd_segment_summary(x, dt, A, B, chunk_size, workspace=workspace,
                                       stream=stream)
        payload = torch.cat([s_r.reshape(-1), d_r.reshape(-1)])
    else:  # no later segment needs the last one's summary
        payload = torch.zeros(n_state + b * H, device=x.device, dtype=torch.float32)
    # the exchange: CUDA tensors for NCCL, host tensors for other backends
    on_dev = dist.get_backend(group) == "nccl"
    if not on_dev and payload.is_cuda:
        s = stream if stream is not None else torch.cuda.current_stream(x.device)
        s.synchronize()
        payload = payload.cpu()
    parts = [torch.empty_like(payload) for _ in range(R)]
    dist.all_gather(parts, payload, group=group)
    allp = torch.stack(parts).to(x.device, non_blocking=False)
    seg_states = allp[:, :n_state].reshape(R, b, H, P, Sd).contiguous()
    seg_decays = allp[:, n_state:].reshape(R, b, H).contiguous()
    h_in = ssd_carry_in(seg_states, seg_decays, r, initial_state=initial_state, stream=stream)
    return ssd_fwd(x, dt, A, B, C, D, chunk_size=chunk_size, initial_state=h_in,
                   return_final_state=True, return_chunk_states=return_chunk_states,
                   workspace=workspace, stream=stream)


def ssd_stream_status(stream=None) -> int:
    """Synchronize the stream and read/clear the kernels' status word."""
    return int(_lib.load().ssd_stream_status(_stream(stream)))
