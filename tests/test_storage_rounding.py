"""Pins of the rounding bound that the parity tests add for results stored in
a narrower type (bf16, fp16, fp8 e4m3 / e5m2 states and checkpoints): it must
hold for round-to-nearest-even into each type, checked here against torch's
own conversions of values across the normal and subnormal ranges, and it must
not be loose: a one-ulp error must break it somewhere.  CPU only."""
import numpy as np
import pytest
import torch

from gdn_testlib import STORED, rounding_bound


def _finite_max(dtype):
    return float(torch.finfo(dtype).max)


@pytest.mark.parametrize("dtype", list(STORED))
def test_bound_holds_for_round_to_nearest(dtype):
    gen = torch.Generator().manual_seed(7)
    tiny = float(torch.finfo(dtype).tiny)
    # magnitudes from deep in the subnormal range up to half the largest finite value
    mags = torch.exp(torch.empty(20000).uniform_(np.log(tiny / 64), np.log(_finite_max(dtype) / 2), generator=gen))
    x = (mags * torch.sign(torch.randn(20000, generator=gen))).to(torch.float64)
    r = x.to(torch.float32).to(dtype).to(torch.float64)
    assert torch.isfinite(r).all()
    err = (r - x).abs().numpy()
    assert (err <= rounding_bound(x.numpy(), dtype) * (1 + 1e-12)).all()


@pytest.mark.parametrize("dtype", list(STORED))
def test_bound_is_tight(dtype):
    # a value halfway between two neighbours in the normal range rounds by exactly the bound's relative part:
    # a bound of half the size would fail there
    m, _ = STORED[dtype]
    x = np.float64(1.0 + 2.0 ** -(m + 1))  # halfway between 1 and 1 + 2^-m
    r = float(torch.tensor(x).to(torch.float32).to(dtype).to(torch.float64))
    assert abs(r - x) == pytest.approx(2.0 ** -(m + 1))
    assert abs(r - x) > 0.5 * (rounding_bound(np.array([x]), dtype)[0] - STORED[dtype][1])
