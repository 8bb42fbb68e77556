"""C-ABI checks that need no GPU: the library loads, exports every entry point
declared in include/ssd.h, and rejects each class of invalid argument on the
host with the documented status before launching anything."""
import ctypes
import os
import re

import pytest

from state_space_sequence_cumsum_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssd.h")


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssd_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(7):
        assert lib.ssd_status_string(code)
    assert b"timed out" in lib.ssd_status_string(_lib.SSD_ERR_TIMEOUT)


FAKE = ctypes.c_void_p(0x10000)       # aligned, never dereferenced (validation fails first)
MISALIGNED = ctypes.c_void_p(0x10008)


def cumsum(lib, d, T, dt=FAKE, A=FAKE, G=FAKE, dtT=None):
    return lib.ssd_chunk_cumsum(dt, A, G, dtT, d, T, None)


@pytest.mark.parametrize("dims,T,expect", [
    ((0, 16, 2, 8, 8, 1), 16, _lib.SSD_ERR_INVALID_ARG),      # batch 0
    ((1, -1, 2, 8, 8, 1), 16, _lib.SSD_ERR_INVALID_ARG),      # negative seqlen
    ((1, 16, 3, 8, 8, 2), 16, _lib.SSD_ERR_INVALID_ARG),      # H % G != 0
    ((1, 16, 2, 8, 8, 1), 0, _lib.SSD_ERR_INVALID_ARG),       # stages need T > 0
    ((1, 16, 2, 8, 8, 1), 257, _lib.SSD_ERR_UNSUPPORTED),     # T > 256
    ((1, 16, 2, 300, 8, 1), 16, _lib.SSD_ERR_UNSUPPORTED),    # P > 256
    ((1, 16, 2, 8, 600, 1), 16, _lib.SSD_ERR_UNSUPPORTED),    # S > 512
    ((70000, 16, 2, 8, 8, 1), 16, _lib.SSD_ERR_UNSUPPORTED),  # batch beyond grid
])
def test_invalid_dims(lib, dims, T, expect):
    d = _lib.dims(*dims)
    assert lib.ssd_state_pass(FAKE, FAKE, FAKE, FAKE, None, None, None, d, 0, T, None) == expect
    assert lib.ssd_chunk_out(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, d, 0, T,
                             None) == expect


def test_null_and_misaligned_pointers(lib):
    before = lib.ssd_launch_count()
    d = _lib.dims(1, 32, 2, 8, 8, 1)
    assert cumsum(lib, d, 16, dt=None) == _lib.SSD_ERR_INVALID_ARG
    assert cumsum(lib, d, 16, A=None) == _lib.SSD_ERR_INVALID_ARG
    assert cumsum(lib, d, 16, G=MISALIGNED) == _lib.SSD_ERR_ALIGNMENT
    assert cumsum(lib, d, 16, dtT=MISALIGNED) == _lib.SSD_ERR_ALIGNMENT
    assert lib.ssd_chunk_out(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, d, 0, 16,
                             None) == _lib.SSD_ERR_INVALID_ARG  # chunk_states required
    assert lib.ssd_state_pass(FAKE, FAKE, FAKE, FAKE, MISALIGNED, None, None, d, 0, 16,
                              None) == _lib.SSD_ERR_ALIGNMENT
    assert lib.ssd_launch_count() == before  # rejected calls launch nothing


def test_bad_dtype(lib):
    d = _lib.dims(1, 32, 2, 8, 8, 1)
    assert lib.ssd_state_pass(FAKE, FAKE, FAKE, FAKE, None, None, None, d, 7, 16,
                              None) == _lib.SSD_ERR_INVALID_ARG


def test_fwd_workspace_checks(lib):
    d = _lib.dims(2, 300, 4, 16, 32, 2)
    need = lib.ssd_fwd_workspace_size(d, 0, 64, 0)
    assert need > 0 and need % 256 == 0
    args = [FAKE] * 6 + [None, FAKE, None, None, d, 0, 64]
    assert lib.ssd_fwd(*args, None, need, None) == _lib.SSD_ERR_WORKSPACE
    assert lib.ssd_fwd(*args, FAKE, need - 256, None) == _lib.SSD_ERR_WORKSPACE
    assert lib.ssd_fwd(*args, ctypes.c_void_p(0x10010), need, None) == _lib.SSD_ERR_WORKSPACE


def test_workspace_size_grows_with_problem(lib):
    # one head per group: the cumsum + fused path, whose G / dt_t buffers grow with L
    small = lib.ssd_fwd_workspace_size(_lib.dims(1, 1024, 8, 64, 128, 8), 0, 128, 0)
    big = lib.ssd_fwd_workspace_size(_lib.dims(1, 4096, 8, 64, 128, 8), 0, 128, 0)
    assert big > small > 0
    assert lib.ssd_fwd_workspace_size(_lib.dims(0, 1, 1, 1, 1, 1), 0, 64, 0) == 0
    # asking for caller-owned chunk states never needs more workspace
    d = _lib.dims(1, 4096, 8, 64, 128, 1)
    assert lib.ssd_fwd_workspace_size(d, 0, 128, 1) <= lib.ssd_fwd_workspace_size(d, 0, 128, 0)


def test_auto_chunk_size_is_supported(lib):
    for L in (1, 64, 1000, 4096, 262144):
        T = lib.ssd_fwd_chosen_chunk_size(_lib.dims(1, L, 8, 64, 128, 1), 0)
        assert T in (64, 128, 256)


def test_auto_chunk_size_is_fixed_by_the_first_query(lib):
    """Without a timed call, the first query fixes the static choice; it then
    never changes, and the chunk_size-0 workspace becomes that choice's."""
    for code, want in ((0, 128), (1, 128)):
        d = _lib.dims(3, 777, 6, 64, 128, 3)  # a shape no other test uses
        before = lib.ssd_fwd_workspace_size(d, code, 0, 0)
        assert lib.ssd_fwd_chunk_size_was_timed(d, code) == 0
        T = lib.ssd_fwd_chosen_chunk_size(d, code)
        assert T == want
        assert lib.ssd_fwd_chosen_chunk_size(d, code) == T
        assert lib.ssd_fwd_chunk_size_was_timed(d, code) == 0
        after = lib.ssd_fwd_workspace_size(d, code, 0, 0)
        assert after == lib.ssd_fwd_workspace_size(d, code, T, 0)
        # before the choice was fixed the size covered every candidate
        assert before >= after
        assert lib.ssd_fwd_path(d, code, 0, 0) == lib.ssd_fwd_path(d, code, T, 0)
    # f32 sequences of at most 64 tokens take 64
    assert lib.ssd_fwd_chosen_chunk_size(_lib.dims(1, 50, 2, 16, 16, 1), 1) == 64
    # invalid arguments
    assert lib.ssd_fwd_chosen_chunk_size(_lib.dims(0, 50, 2, 16, 16, 1), 0) == 0
    assert lib.ssd_fwd_chosen_chunk_size(_lib.dims(1, 50, 2, 16, 16, 1), 7) == 0


def test_decode_step_validation(lib):
    before = lib.ssd_launch_count()
    d1 = _lib.dims(2, 1, 4, 16, 32, 2)
    args = lambda si=FAKE, so=FAKE, y=FAKE, x=FAKE: (x, FAKE, FAKE, FAKE, FAKE, FAKE, si, so, y)
    # more than one token
    assert lib.ssd_decode_step(*args(), _lib.dims(2, 2, 4, 16, 32, 2), 0, None) == \
        _lib.SSD_ERR_INVALID_ARG
    assert lib.ssd_decode_step(*args(x=None), d1, 0, None) == _lib.SSD_ERR_INVALID_ARG
    # element alignment only: 8-byte offsets are fine, odd addresses are not
    assert lib.ssd_decode_step(*args(y=ctypes.c_void_p(0x10001)), d1, 0, None) == \
        _lib.SSD_ERR_ALIGNMENT
    assert lib.ssd_decode_step(*args(si=ctypes.c_void_p(0x10002), so=ctypes.c_void_p(0x10002)),
                               d1, 1, None) == _lib.SSD_ERR_ALIGNMENT
    assert lib.ssd_decode_step(*args(so=None), d1, 0, None) == _lib.SSD_ERR_INVALID_ARG
    assert lib.ssd_decode_step(*args(), d1, 5, None) == _lib.SSD_ERR_INVALID_ARG  # dtype
    # partly overlapping state buffers (the same buffer is fine: in place)
    assert lib.ssd_decode_step(*args(si=FAKE, so=ctypes.c_void_p(0x10000 + 256)), d1, 0,
                               None) == _lib.SSD_ERR_INVALID_ARG
    assert lib.ssd_launch_count() == before


def test_bwd_validation(lib):
    before = lib.ssd_launch_count()
    d = _lib.dims(2, 100, 4, 16, 32, 2)
    need = lib.ssd_bwd_workspace_size(d, 0)
    assert need > 0 and need % 256 == 0
    args = [FAKE] * 6 + [None, FAKE, None] + [FAKE] * 6 + [None, d, 0]
    assert lib.ssd_bwd(*args, None, need, None) == _lib.SSD_ERR_WORKSPACE
    assert lib.ssd_bwd(*args, FAKE, need - 256, None) == _lib.SSD_ERR_WORKSPACE
    # headdim above 64 is not served by the backward
    big = _lib.dims(2, 100, 4, 128, 32, 2)
    a2 = [FAKE] * 6 + [None, FAKE, None] + [FAKE] * 6 + [None, big, 0]
    assert lib.ssd_bwd(*a2, FAKE, 1 << 40, None) == _lib.SSD_ERR_UNSUPPORTED
    assert lib.ssd_launch_count() == before


def test_gated_rmsnorm_validation(lib):
    before = lib.ssd_launch_count()
    f = lib.ssd_gated_rmsnorm
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 96, 40, 1e-5, 0, None) == _lib.SSD_ERR_INVALID_ARG  # 96 % 40
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 96, 32, -1.0, 0, None) == _lib.SSD_ERR_INVALID_ARG  # eps < 0
    assert f(None, FAKE, FAKE, FAKE, 4, 96, 32, 1e-5, 0, None) == _lib.SSD_ERR_INVALID_ARG
    assert f(FAKE, ctypes.c_void_p(0x10001), FAKE, FAKE, 4, 96, 32, 1e-5, 0, None) == \
        _lib.SSD_ERR_ALIGNMENT
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 96, 32, 1e-5, 9, None) == _lib.SSD_ERR_INVALID_ARG
    assert lib.ssd_launch_count() == before


def test_fwd_host_validation(lib):
    """ssd_fwd_host checks its arguments and workspace on the host before any
    copy or launch (a rejected call launches nothing)."""
    before = lib.ssd_launch_count()
    d = _lib.dims(2, 3000, 4, 64, 128, 2)
    need = lib.ssd_fwd_host_workspace_size(d, 0, 128)
    assert need > 0 and need % 256 == 0
    # the parts and the slots grow with the sequence
    assert lib.ssd_fwd_host_workspace_size(_lib.dims(2, 30000, 4, 64, 128, 2), 0, 128) > need
    # invalid dims / dtype / chunk size: no size
    assert lib.ssd_fwd_host_workspace_size(_lib.dims(0, 3000, 4, 64, 128, 2), 0, 128) == 0
    assert lib.ssd_fwd_host_workspace_size(d, 7, 128) == 0
    assert lib.ssd_fwd_host_workspace_size(d, 0, 512) == 0
    host = [FAKE] * 6  # x, dt, A, B, C, D
    ok_tail = [None, FAKE, None, d, 0, 128]
    # a required input missing
    for k in range(6):
        args = list(host)
        args[k] = None
        assert lib.ssd_fwd_host(*args, *ok_tail, FAKE, need, None) == _lib.SSD_ERR_INVALID_ARG
    # no y for a non-empty sequence
    assert lib.ssd_fwd_host(*host, None, None, None, d, 0, 128, FAKE, need, None) == _lib.SSD_ERR_INVALID_ARG
    # workspace missing, short or not 256-byte aligned
    assert lib.ssd_fwd_host(*host, *ok_tail, None, need, None) == _lib.SSD_ERR_WORKSPACE
    assert lib.ssd_fwd_host(*host, *ok_tail, FAKE, need - 256, None) == _lib.SSD_ERR_WORKSPACE
    assert lib.ssd_fwd_host(*host, *ok_tail, ctypes.c_void_p(0x10010), need, None) == _lib.SSD_ERR_WORKSPACE
    assert lib.ssd_launch_count() == before
