"""The accurate exponential of the fp32 path (sscan_exp2_accurate) against the exact 2^x.

The fp32 scan re-anchors the decay over every chunk on this exponential, so it has to be
accurate (about one ulp) and, above all, unbiased: a factor that is consistently low or high
would compound over a state's memory of up to thousands of steps.
"""
import numpy as np
import pytest
import torch

from selective_state_space_158_b300 import binding

pytestmark = pytest.mark.gpu


def test_exp2_accurate_within_two_ulp_and_unbiased():
    g = torch.Generator(device="cuda:0")
    g.manual_seed(17)
    dense = torch.linspace(-40.0, 40.0, 2_000_001, device="cuda:0")
    small = -torch.rand(1_000_000, generator=g, device="cuda:0") * 0.2  # chunk decays dt*A*S
    tiny = -torch.rand(1_000_000, generator=g, device="cuda:0") * 1e-3
    x = torch.cat([dense, small, tiny]).contiguous()
    y = binding.exp2_accurate(x).double().cpu().numpy()
    xd = x.double().cpu().numpy()
    ref = np.exp2(xd)
    rel = (y - ref) / ref
    assert np.max(np.abs(rel)) <= 2.4e-7, np.max(np.abs(rel))  # two fp32 ulp at [1, 2)
    assert abs(float(np.mean(rel))) <= 2e-9, np.mean(rel)
    # the slow-decay region where compounding matters: unbiased there too
    sel = xd[-2_000_000:]
    r2 = rel[-2_000_000:]
    assert abs(float(np.mean(r2))) <= 5e-9 and sel.max() <= 0.0


def test_exp2_accurate_clamps_and_handles_empty():
    x = torch.tensor([-1000.0, -125.0, 0.0, 1.0, 125.0, 1000.0], device="cuda:0")
    y = binding.exp2_accurate(x).cpu().numpy().astype(np.float64)
    want = np.exp2(np.array([-125.0, -125.0, 0.0, 1.0, 125.0, 125.0]))
    assert np.all(np.abs(y - want) / want <= 2.4e-7)
    assert binding.exp2_accurate(torch.empty(0, device="cuda:0")).numel() == 0
