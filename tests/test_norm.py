"""GPU parity of the gated RMS norm (ssd_gated_rmsnorm) against the oracle.

f32 arithmetic on exactly widened inputs: f32 calls within 1e-4 * rms; bf16
calls return the f32 result rounded to bf16, held element by element to the
rounding bound 2^-8 |oracle| + 1e-4 * rms."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import rel_err
import state_space_sequence_cumsum_gb300 as ssd

pytestmark = pytest.mark.gpu


def check(out, ref, dtype):
    if dtype == torch.float32:
        assert rel_err(out, ref) <= 1e-4
    else:
        g = out.detach().to("cpu", torch.float64).numpy()
        rms = float(np.sqrt(np.mean(ref * ref)))
        assert np.max(np.abs(g - ref) - (2.0 ** -8 * np.abs(ref) + 1e-4 * rms)) <= 0.0


@pytest.mark.parametrize("shape,gs,dtype", [
    ((4, 64, 80 * 64), None, torch.bfloat16),   # tokens of the 2.7B layer, one group
    ((3, 17, 8 * 64), 64, torch.bfloat16),      # per-head groups
    ((2, 33, 4 * 32), 32, torch.float32),
    ((5, 96), 24, torch.float32),               # 24 % 8 != 0 for bf16 vectors
    ((7, 40), 20, torch.bfloat16),              # scalar path
])
def test_gated_rmsnorm_matches_oracle(shape, gs, dtype):
    g = torch.Generator().manual_seed(3)
    y = torch.randn(shape, generator=g).to(dtype)
    z = (2.0 * torch.randn(shape, generator=g)).to(dtype)
    w = 1.0 + 0.1 * torch.randn(shape[-1], generator=g)
    out = ssd.ssd_gated_rmsnorm(y.cuda(), z.cuda(), w.cuda(), eps=1e-5, group_size=gs)
    torch.cuda.synchronize()
    ref = oracle.gated_rmsnorm(y, z, w, 1e-5, shape[-1] if gs is None else gs)
    check(out, ref, dtype)


def test_gated_rmsnorm_in_place_on_scan_output():
    """The scan's y [B, L, H, P] viewed as [B*L, H*P], normalised in place."""
    B, L, H, P = 2, 130, 8, 64
    g = torch.Generator().manual_seed(4)
    y = torch.randn((B, L, H, P), generator=g).to(torch.bfloat16)
    z = torch.randn((B, L, H, P), generator=g).to(torch.bfloat16)
    w = torch.ones(H * P)
    ref = oracle.gated_rmsnorm(y.reshape(B * L, H * P), z.reshape(B * L, H * P), w, 1e-6, H * P)
    yd = y.cuda()
    out = ssd.ssd_gated_rmsnorm(yd.view(B * L, H * P), z.cuda().view(B * L, H * P), w.cuda(),
                                eps=1e-6, out=yd.view(B * L, H * P))
    torch.cuda.synchronize()
    assert out.data_ptr() == yd.data_ptr()
    check(yd.view(B * L, H * P), ref, torch.bfloat16)
