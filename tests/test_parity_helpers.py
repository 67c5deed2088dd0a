"""CPU checks of the parity helpers' bf16 rounding allowance."""

import numpy as np
import torch

from tests.parity import half_ulp_bf16


def test_half_ulp_bounds_bf16_rounding():
    """Round-to-nearest bf16 moves x by at most half_ulp_bf16(x), over many magnitudes.
    x is fp32, as the kernel's accumulator is, so the conversion rounds once."""
    g = torch.Generator().manual_seed(0)
    x = torch.randn(200_000, generator=g) * torch.exp2(torch.randint(-20, 20, (200_000,), generator=g).float())
    err = (x.to(torch.bfloat16).double() - x.double()).abs().numpy()
    assert np.all(err <= half_ulp_bf16(x.double().numpy()))


def test_half_ulp_is_tight():
    """The bound is reached: ties of round-to-nearest-even sit exactly half an ulp away."""
    for e in (-3, 0, 2, 5):
        x = np.array([2.0 ** e * (1 + 2.0 ** -8)])   # halfway between 2^e and the next bf16 value
        err = abs(float(torch.tensor(x).to(torch.bfloat16).double()) - x[0])
        assert err == half_ulp_bf16(x)[0] == 2.0 ** (e - 8)
    assert half_ulp_bf16(np.array([0.0, -4.075]))[0] == 0.0
    assert half_ulp_bf16(np.array([-4.075]))[0] == 2.0 ** -6
