"""The time-lane kernel (time_scan = 1): a warp scans one channel over time, its 32 lanes each
run a stretch of 8 steps from a zero state, the lanes' aggregates are composed in order with
(a2, b2) o (a1, b1) = (a2 a1, a2 b1 + b2), and every lane runs its steps again from its true
start state with the readout. Compared element by element with the fp64 oracle over whole
tensors: ragged sequence ends (L not a multiple of the 256-step chunk) and channel tiles (D not a
multiple of 8), every optional operand, time segments joined by the chunk carry, an initial
state (also in place), the first-order factor, N < 16, bitwise repeatability, the segment
carry's timeout path, and agreement with the lane kernel on a few-channel long sequence."""
import pytest
import torch

from parity import assert_within, compare, oracle_full
from selective_state_space_158_b300 import binding
from selective_state_space_158_b300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _run(x, softplus=True, h0=None, euler=False, h_last=None):
    y, h = binding.fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x.get("D"), x.get("z"),
                       x.get("delta_bias"), softplus=softplus, h0=h0, euler=euler,
                       h_last=h_last)
    assert binding.device_error() == 0
    return y, h


def _check(w, x=None, softplus=True, h0=None, euler=False, what=""):
    x = x if x is not None else make_inputs(w, device=DEV)
    y, h = _run(x, softplus, h0, euler)
    yr, hr, ym = oracle_full(x, softplus, h0=h0, euler=euler)
    res = compare(y, h, yr, hr, w.io, y_mag=ym)
    assert_within(res, w.io, what)
    return y, h


def _h0(w, seed=7):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return torch.randn((w.batch, w.dim, w.N), generator=g, device=DEV, dtype=torch.float32)


@pytest.mark.parametrize("segments", [1, 3, 0])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_ragged_shapes_and_segments(io, segments, tune):
    tune(time_scan=1, segments=segments)
    base = WORKLOADS["fp32"] if io == "f32" else WORKLOADS["bf16"]
    w = base.replace(batch=2, L=3001, dim=24 if io == "f32" else 40)
    _check(w, what=f"time lanes {io} segments={segments}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_optional_operands_off_and_softplus_off(io, tune):
    tune(time_scan=1, segments=2)
    base = WORKLOADS["tiny"] if io == "f32" else WORKLOADS["long"]  # no gate; long: no D either
    w = base.replace(batch=1, L=3000, dim=16)
    _check(w, what=f"time lanes, no gate {io}")
    x = make_inputs(w, device=DEV)
    x["delta"] = (x["delta"].float().abs() * 0.05).to(x["u"].dtype)  # positive steps as given
    x["delta_bias"] = None
    _check(w, x=x, softplus=False, what=f"time lanes, softplus off {io}")


@pytest.mark.parametrize("segments", [1, 4])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_initial_state_in_place_and_first_order(io, segments, tune):
    tune(time_scan=1, segments=segments)
    base = WORKLOADS["fp32"] if io == "f32" else WORKLOADS["bf16"]
    w = base.replace(batch=1, L=2100, dim=16)
    h0 = _h0(w)
    _check(w, h0=h0, what=f"time lanes h0 {io} segments={segments}")
    x = make_inputs(w, device=DEV)
    hl = h0.clone()  # h0 aliases h_last: continued in place
    y, h = _run(x, h0=hl, h_last=hl)
    yr, hr, ym = oracle_full(x, h0=h0)
    assert_within(compare(y, h, yr, hr, w.io, y_mag=ym), w.io, "time lanes in place")
    x["delta"] = (x["delta"].float().abs() * 0.02).to(x["u"].dtype)
    x["delta_bias"] = None
    _check(w, x=x, softplus=False, h0=h0, euler=True, what=f"time lanes first order {io}")


def test_fewer_states_than_sixteen(tune):
    tune(time_scan=1, segments=3)
    w = WORKLOADS["bf16"].replace(batch=1, L=2600, dim=8, N=5)
    _check(w, what="time lanes N=5")


def test_bitwise_repeatable_and_agrees_with_lane_kernel(tune):
    """Two calls give identical bits; the lane kernel gives the same results within the parity
    bounds on a long sequence with few channels (the time lanes' regime)."""
    w = WORKLOADS["long"].replace(batch=1, L=1 << 16, dim=16)
    x = make_inputs(w, device=DEV)
    tune(time_scan=1)
    y1, h1 = _run(x)
    y2, h2 = _run(x)
    assert torch.equal(y1, y2) and torch.equal(h1, h2)
    yr, hr, ym = oracle_full(x)
    assert_within(compare(y1, h1, yr, hr, w.io, y_mag=ym), w.io, "time lanes, long narrow")
    tune(time_scan=2)
    y3, h3 = _run(x)
    assert_within(compare(y3, h3, yr, hr, w.io, y_mag=ym), w.io, "lane kernel, long narrow")


def test_segment_timeout_reports_status_and_context_survives(tune):
    tune(time_scan=1, segments=3, test_skip_publish=0)
    w = WORKLOADS["fp32"].replace(batch=1, L=2000, dim=8)
    x = make_inputs(w, device=DEV)
    binding.fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"])
    assert binding.device_error() == 4  # SSCAN_ERR_CARRY_TIMEOUT
    assert binding.device_error() == 0
    tune(time_scan=1, segments=3)
    _check(w, x=x, what="time lanes after timeout")
