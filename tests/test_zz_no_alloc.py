"""ssd_fwd_noalloc: the forward for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (they run inside an allocator callback,
or a host framework owns every device allocation), so they cannot provide
ssd_fwd's workspace.  ssd_fwd_noalloc uses a fixed scratch array inside the
library instead.  This test calls it through the C ABI and checks, on two
calls in a row, that it reproduces ssd_fwd within the parity tolerance used
by every GPU test (2e-2 of the output's rms for bf16 inputs, 1e-4 for f32)
-- in fact bit for bit, since the same kernels and plan run -- and that
sizes beyond the scratch array are refused before any launch.  Before the
calls that are checked, a call on other inputs leaves its own values in the
scratch array, so a kernel that read scratch before writing it would show.
The cases cover the head-pair path (one CTA per pair, prefilled segments,
and the wrap plan whose sequences hand states from CTA to CTA), the one-head
fused path at dstate 256 (prefilled segments, and hand-off segments when there
are more sequences than SMs), the staged dstate-512 path (taken when chunk
states are asked for) and the f32 path.

The file is named so pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from parity_util import TOL, case_inputs, to_gpu
import state_space_sequence_cumsum_gb300 as ssd
from state_space_sequence_cumsum_gb300 import _lib

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, g, y, fin, T, dtype_code, states=None):
    b, L, H, P = g["x"].shape
    d = _lib.dims(b, L, H, P, g["B"].shape[3], g["B"].shape[2])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.ssd_fwd_noalloc(_p(g["x"]), _p(g["dt"]), _p(g["A"]), _p(g["B"]), _p(g["C"]),
                               _p(g["D"]), _p(g["init"]), _p(y), _p(fin), _p(states), d,
                               dtype_code, T, stream)


def _max_rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.max(np.abs(a - b)) / max(np.sqrt(np.mean(b * b)), 1e-30))


@pytest.mark.parametrize("shape,dtype,want_states", [
    ((2, 777, 8, 64, 128, 2, 256), torch.bfloat16, False),   # head pairs, one CTA per pair
    ((1, 4096, 2, 64, 128, 1, 128), torch.bfloat16, False),  # head pairs, prefilled segments
    ((1, 300, 320, 64, 64, 1, 128), torch.bfloat16, False),  # head pairs, wrap plan (160 pairs)
    ((1, 1000, 3, 64, 256, 1, 128), torch.bfloat16, False),  # one-head fused, dstate 256, prefilled
    ((1, 600, 160, 64, 256, 1, 128), torch.bfloat16, False),  # one-head fused, hand-off segments
    ((1, 600, 2, 64, 512, 1, 128), torch.bfloat16, True),    # staged, dstate 512, chunk states
    ((1, 300, 3, 32, 48, 1, 64), torch.float32, False),      # f32 CUDA cores
])
def test_noalloc_matches_ssd_fwd_twice(shape, dtype, want_states):
    B, L, H, P, S, G, T = shape
    lib = _lib.load()
    inp = case_inputs(B, L, H, P, S, G, T, dtype=dtype, init="randn", seed=L)
    g = to_gpu(inp)
    y_ref, f_ref, st_ref = ssd.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], T,
                                       initial_state=g["init"],
                                       return_chunk_states=want_states)
    code = _lib.SSD_BF16 if dtype == torch.bfloat16 else _lib.SSD_F32
    # leave another call's values in the scratch array first
    other = to_gpu(case_inputs(B, L, H, P, S, G, T, dtype=dtype, init="randn", seed=L + 1))
    assert _noalloc(lib, other, torch.empty_like(g["x"]), torch.empty_like(f_ref), T, code,
                    None if st_ref is None else torch.empty_like(st_ref)) == _lib.SSD_OK
    for _ in range(2):  # the scratch array keeps the previous call's contents
        y = torch.full_like(g["x"], float("nan"))
        fin = torch.full_like(f_ref, float("nan"))
        st = None if st_ref is None else torch.full_like(st_ref, float("nan"))
        assert _noalloc(lib, g, y, fin, T, code, st) == _lib.SSD_OK
        assert ssd.ssd_stream_status() == 0
        assert _max_rel(y, y_ref) <= TOL[dtype]
        assert _max_rel(fin, f_ref) <= TOL[dtype]
        # the same kernels and plan as ssd_fwd: the same bits
        assert torch.equal(y, y_ref)
        assert torch.equal(fin, f_ref)
        if st is not None:
            assert torch.equal(st, st_ref)


def test_noalloc_refuses_sizes_beyond_its_scratch():
    lib = _lib.load()
    big = _lib.dims(64, 262144, 64, 64, 128, 1)  # G_cum + dt_t alone need 8 GiB
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: rejected before any launch
    before = lib.ssd_launch_count()
    st = lib.ssd_fwd_noalloc(fake, fake, fake, fake, fake, fake, None, fake, None, None, big,
                             _lib.SSD_BF16, 128, None)
    assert st == _lib.SSD_ERR_UNSUPPORTED
    assert lib.ssd_launch_count() == before
