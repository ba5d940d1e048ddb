"""Degenerate steps and size limits, against the fp64 oracle over whole tensors:

* a vanishing step (softplus of a very negative input, dt ~ 1e-26): every decay factor is 1 and
  every input term 0, so the state stays at h0 and y = (C . h0 + D u) SiLU(z) at every step
  ("架构变体：Mamba/SSM": Delta -> 0 leaves the state unchanged); in the lane kernel and in the
  time lanes, split into segments;
* a very large step (dt = 30): the state forgets everything before the current step;
* more batch rows than a grid dimension holds (65537, bf16: the plain-load kernel), and 32768
  channels in one batch row (one lane per channel, 128 CTAs)."""
import pytest
import torch

from parity import assert_within, compare, oracle_full
from selective_state_space_158_b300 import binding
from selective_state_space_158_b300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _h0(w, seed=3):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return torch.randn((w.batch, w.dim, w.N), generator=g, device=DEV, dtype=torch.float32)


def _check(w, x, h0=None, what=""):
    y, h = binding.fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x.get("D"), x.get("z"),
                       x.get("delta_bias"), h0=h0)
    assert binding.device_error() == 0
    yr, hr, ym = oracle_full(x, h0=h0)
    assert_within(compare(y, h, yr, hr, w.io, y_mag=ym), w.io, what)
    return y, h


@pytest.mark.parametrize("time_scan", [2, 1])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_vanishing_step_keeps_the_initial_state(io, time_scan, tune):
    tune(time_scan=time_scan, segments=3)
    base = WORKLOADS["fp32"] if io == "f32" else WORKLOADS["bf16"]
    w = base.replace(batch=2, L=3000, dim=16)
    x = make_inputs(w, device=DEV)
    x["delta"] = torch.full_like(x["delta"], -60.0)
    x["delta_bias"] = None
    h0 = _h0(w)
    y, h = _check(w, x, h0=h0, what=f"vanishing step {io} time_scan={time_scan}")
    assert torch.allclose(h, h0, rtol=1e-6, atol=0)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_large_step_forgets(io):
    base = WORKLOADS["fp32"] if io == "f32" else WORKLOADS["bf16"]
    w = base.replace(batch=2, L=700, dim=64)
    x = make_inputs(w, device=DEV)
    x["delta"] = torch.full_like(x["delta"], 30.0)
    x["delta_bias"] = None
    _check(w, x, h0=_h0(w), what=f"large step {io}")


def test_more_batch_rows_than_a_grid_dimension():
    """bf16 io: with 8.4M fp32 end states of three steps each, the survey scale's max over
    near-cancelled entries reflects fp32 rounding of their terms rather than the path under
    test (the same effect as for fp32 y, reading 10)."""
    w = WORKLOADS["bf16"].replace(batch=65537, L=40, dim=8)
    x = make_inputs(w, device=DEV)
    _check(w, x, what="65537 batch rows")


def test_many_channels_in_one_row():
    w = WORKLOADS["bf16"].replace(batch=1, L=40, dim=32768)
    x = make_inputs(w, device=DEV)
    _check(w, x, what="32768 channels")
