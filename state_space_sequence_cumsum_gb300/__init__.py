"""GB300 (sm_103a) Mamba-2 chunked SSD forward.

The compute lives in ``libssd.so`` (hand-written CUDA behind the C ABI in
``include/ssd.h``); this package is its thin binding.  Importing it does not
load the library; the first call does, and raises if the library cannot be
built or loaded (there is no CPU fallback).
"""
from .ssd import (SsdError, SsdFunction, Workspace, ssd_bwd, ssd_chunk_cumsum,  # noqa: F401
                  ssd_chunk_out, ssd_decode_step, ssd_fwd, ssd_fwd_host, ssd_gated_rmsnorm,
                  ssd_fwd_chosen_chunk_size, ssd_fwd_chunk_size_was_timed, ssd_fwd_path,
                  ssd_fwd_plan, ssd_fwd_staged, ssd_fwd_workspace_size, ssd_state_out,
                  ssd_state_pass, ssd_status_string, ssd_stream_status, ssd_segment_summary,
                  ssd_carry_in, ssd_fwd_context_parallel)
from ._build import build  # noqa: F401
