"""ctypes binding of ``libssd.so`` (declared in ``include/ssd.h``).

Argument marshalling only: every step of the SSD forward runs in the CUDA
kernels behind the C ABI.  There is no CPU fallback; if the library is
missing or cannot be built, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

SSD_OK = 0
SSD_ERR_INVALID_ARG = 1
SSD_ERR_UNSUPPORTED = 2
SSD_ERR_ALIGNMENT = 3
SSD_ERR_CUDA = 4
SSD_ERR_TIMEOUT = 5
SSD_ERR_WORKSPACE = 6
SSD_BF16 = 0
SSD_F32 = 1

# Every entry point include/ssd.h declares (checked by the tests).
EXPORTS = ("ssd_chunk_cumsum", "ssd_state_pass", "ssd_chunk_out", "ssd_state_out",
           "ssd_state_out_workspace_size",
           "ssd_fwd_path", "ssd_fwd_workspace_size", "ssd_fwd", "ssd_fwd_noalloc",
           "ssd_fwd_host", "ssd_fwd_host_workspace_size",
           "ssd_fwd_chosen_chunk_size", "ssd_fwd_chunk_size_was_timed", "ssd_decode_step",
           "ssd_bwd", "ssd_bwd_workspace_size",
           "ssd_gated_rmsnorm", "ssd_segment_summary", "ssd_segment_summary_workspace_size",
           "ssd_carry_in",
           "ssd_launch_count", "ssd_status_string", "ssd_stream_status")
PATH_NAMES = {0: "staged-cuda-cores", 1: "staged-tensor-cores", 2: "fused-tensor-cores",
              3: "fused-pair-tensor-cores"}


class ssd_dims_t(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64),
                ("nheads", ctypes.c_int64), ("headdim", ctypes.c_int64),
                ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64)]


class SsdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) the CUDA library; raise if impossible."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"CUDA library {_build.LIB} is missing; run __graft_entry__.build()")
        lib = ctypes.CDLL(_build.LIB)
        vp, fp, i32, st = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int
        D = ssd_dims_t
        sig = {
            "ssd_chunk_cumsum": ([fp, fp, fp, fp, D, i32, vp], st),
            "ssd_state_pass": ([vp, vp, fp, fp, fp, fp, fp, D, i32, i32, vp], st),
            "ssd_chunk_out": ([vp, vp, vp, fp, fp, fp, fp, vp, D, i32, i32, vp], st),
            "ssd_state_out": ([vp, vp, vp, fp, fp, fp, fp, vp, fp, fp, D, i32, i32, vp,
                               ctypes.c_size_t, vp], st),
            "ssd_state_out_workspace_size": ([D, i32, i32], ctypes.c_size_t),
            "ssd_fwd_path": ([D, i32, i32, i32], ctypes.c_int),
            "ssd_fwd_workspace_size": ([D, i32, i32, i32], ctypes.c_size_t),
            "ssd_fwd": ([vp, fp, fp, vp, vp, fp, fp, vp, fp, fp, D, i32, i32, vp,
                         ctypes.c_size_t, vp], st),
            "ssd_fwd_noalloc": ([vp, fp, fp, vp, vp, fp, fp, vp, fp, fp, D, i32, i32, vp], st),
            "ssd_fwd_host": ([vp, fp, fp, vp, vp, fp, fp, vp, fp, D, i32, i32, vp,
                              ctypes.c_size_t, vp], st),
            "ssd_fwd_host_workspace_size": ([D, i32, i32], ctypes.c_size_t),
            "ssd_fwd_chosen_chunk_size": ([D, i32], ctypes.c_int),
            "ssd_fwd_chunk_size_was_timed": ([D, i32], ctypes.c_int),
            "ssd_decode_step": ([vp, fp, fp, vp, vp, fp, fp, fp, vp, D, i32, vp], st),
            "ssd_bwd_workspace_size": ([D, i32], ctypes.c_size_t),
            "ssd_gated_rmsnorm": ([vp, vp, fp, vp, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_int64, ctypes.c_float, i32, vp], st),
            "ssd_bwd": ([vp, fp, fp, vp, vp, fp, fp, vp, fp, vp, fp, fp, vp, vp, fp, fp, D, i32,
                         vp, ctypes.c_size_t, vp], st),
            "ssd_segment_summary_workspace_size": ([D, i32, i32], ctypes.c_size_t),
            "ssd_segment_summary": ([vp, fp, fp, vp, fp, fp, D, i32, i32, vp, ctypes.c_size_t,
                                     vp], st),
            "ssd_carry_in": ([fp, fp, fp, i32, i32, fp, D, vp], st),
            "ssd_launch_count": ([], ctypes.c_uint64),
            "ssd_status_string": ([st], ctypes.c_char_p),
            "ssd_stream_status": ([vp], st),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().ssd_status_string(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != SSD_OK:
        raise SsdError(status, where)


def dims(batch, seqlen, nheads, headdim, dstate, ngroups) -> ssd_dims_t:
    return ssd_dims_t(int(batch), int(seqlen), int(nheads), int(headdim), int(dstate),
                      int(ngroups))
