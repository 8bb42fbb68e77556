"""ssd_fwd's choice of kernel path, through the C ABI, on the host alone.

ssd_fwd_path answers from the shape, dtype, chunk size and whether chunk
states are wanted; for a fixed chunk size it touches no GPU, so these run on
the CPU.  They pin which shapes take the head-pair fused kernel, the one-head
fused kernel (dstate up to 256, and 384 / 512 with B / C in dstate blocks),
the staged tensor-core path and the CUDA-core path, and the SSD_FWD_PATH
override.
"""
import pytest

from state_space_sequence_cumsum_gb300 import _lib

BF16, F32 = 0, 1


def path(B, L, H, P, S, G, T, dtype=BF16, want_states=False):
    lib = _lib.load()
    return _lib.PATH_NAMES.get(lib.ssd_fwd_path(_lib.dims(B, L, H, P, S, G), dtype, T, int(want_states)))


@pytest.fixture(autouse=True)
def no_override(monkeypatch):
    monkeypatch.delenv("SSD_FWD_PATH", raising=False)


@pytest.mark.parametrize("S", [64, 128])
def test_head_pairs_for_small_dstate(S):
    assert path(4, 4096, 80, 64, S, 1, 256) == "fused-pair-tensor-cores"
    assert path(4, 4096, 80, 64, S, 1, 128, want_states=True) == "fused-pair-tensor-cores"


def test_one_head_fused_at_dstate_256():
    assert path(2, 32768, 64, 64, 256, 8, 256) == "fused-tensor-cores"
    assert path(2, 32768, 64, 64, 256, 8, 128, want_states=True) == "fused-tensor-cores"


@pytest.mark.parametrize("S", [384, 512])
def test_dstate_blocks_fused_unless_every_chunk_state_is_wanted(S):
    assert path(4, 65536, 64, 64, S, 1, 128) == "fused-tensor-cores"
    assert path(4, 65536, 64, 64, S, 1, 256) == "fused-tensor-cores"
    # every chunk state wanted: the staged path's state pass writes them anyway
    assert path(1, 262144, 32, 64, S, 1, 128, want_states=True) == "staged-tensor-cores"
    # with 256-token chunks the staged chunk output is not on tensor cores
    assert path(1, 262144, 32, 64, S, 1, 256, want_states=True) == "fused-tensor-cores"


def test_override(monkeypatch):
    monkeypatch.setenv("SSD_FWD_PATH", "staged")
    assert path(4, 65536, 64, 64, 512, 1, 128) == "staged-tensor-cores"
    assert path(2, 32768, 64, 64, 256, 8, 256) == "staged-tensor-cores"
    monkeypatch.setenv("SSD_FWD_PATH", "fused")
    assert path(1, 262144, 32, 64, 512, 1, 128, want_states=True) == "fused-tensor-cores"


def test_cuda_cores_outside_the_tensor_core_shapes():
    assert path(1, 4096, 8, 64, 512, 1, 64) == "staged-cuda-cores"      # chunk not whole tiles
    assert path(1, 4096, 8, 64, 128, 1, 128, dtype=F32) == "staged-cuda-cores"
    assert path(1, 4096, 8, 32, 64, 1, 128) == "staged-cuda-cores"      # P 32: no tcgen05 kernel
    # P 128: the tensor-core state pass serves it, the fused passes do not
    assert path(1, 4096, 8, 128, 128, 1, 128) == "staged-tensor-cores"
