"""The parity bound itself: half a bf16 ulp, checked against torch's own
round-to-nearest-even conversion to bfloat16 (no GPU needed)."""
import numpy as np
import torch

from compare import bf16_half_ulp, o_bound, O_MAX_ABS


def test_half_ulp_values():
    # bf16 keeps 8 significant bits: the spacing in [1, 2) is 2^-7
    assert bf16_half_ulp(1.0) == 2.0 ** -8
    assert bf16_half_ulp(1.99) == 2.0 ** -8
    assert bf16_half_ulp(-2.0) == 2.0 ** -7
    assert bf16_half_ulp(0.75) == 2.0 ** -9
    assert bf16_half_ulp(24.0) == 2.0 ** -4
    assert bf16_half_ulp(0.0) == 0.0
    assert o_bound(0.0) == O_MAX_ABS


def test_half_ulp_bounds_bf16_rounding_and_is_reached():
    g = torch.Generator().manual_seed(3)
    # fp32 values (one rounding, fp32 -> bf16, as when a kernel stores O)
    x = (torch.randn(200000, generator=g)
         * torch.exp2(torch.randint(-20, 20, (200000,), generator=g).float())).double()
    r = x.float().to(torch.bfloat16).double()
    err = (r - x).abs().numpy()
    hu = bf16_half_ulp(x.numpy())
    assert np.all(err <= hu * (1 + 1e-12))
    # a midpoint between two bf16 numbers is exactly half an ulp away
    mid = 1.0 + 2.0 ** -8
    assert abs(float(torch.tensor(mid).to(torch.bfloat16)) - mid) == bf16_half_ulp(mid)
