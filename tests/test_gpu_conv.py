"""GPU parity of the causal depthwise Conv1d + SiLU (sscan_conv1d_silu) against the fp64
oracle, alone and feeding the scan."""
import pytest
import torch

import oracle
from parity import assert_within, compare, oracle_full, to_np_io
from selective_state_space_158_b300 import binding
from selective_state_space_158_b300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _conv_ref(x, w, bias, x_prev, silu):
    io = "f32" if x.dtype == torch.float32 else "bf16"
    return oracle.conv1d(to_np_io(x), w.cpu().numpy(),
                         None if bias is None else bias.cpu().numpy(),
                         None if x_prev is None else to_np_io(x_prev), silu=silu, io=io)


@pytest.fixture
def plain_loads(tune):
    tune(conv_plain=1)


def _check_conv(width, io, dim, batch=3, L=200, seed=None):
    g = torch.Generator(device=DEV)
    g.manual_seed(100 + width if seed is None else seed)
    dt = torch.float32 if io == "f32" else torch.bfloat16
    x = torch.randn((batch, L, dim), generator=g, device=DEV).to(dt)
    w = torch.randn((dim, width), generator=g, device=DEV) * 0.5
    bias = torch.randn((dim,), generator=g, device=DEV)
    x_prev = torch.randn((batch, width - 1, dim), generator=g, device=DEV).to(dt)
    for xp, silu in ((None, True), (x_prev, True), (x_prev, False)):
        y = binding.conv1d_silu(x, w, bias, x_prev=xp, silu=silu)
        torch.cuda.synchronize()
        r = _conv_ref(x, w, bias, xp, silu)
        res = compare(y, None, r, None, io)
        assert_within(res, io, f"conv width={width} {io} dim={dim} prev={xp is not None}")


@pytest.mark.parametrize("width", [1, 2, 3, 4, 5, 8, 12])
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("dim", [128, 200, 37])
def test_conv1d_silu(width, io, dim):
    """TMA-staged tiles (width <= 8, 16-byte rows: dim 128 and 200, the latter with a ragged
    channel block) and the general path (width 12, odd dim), with and without the previous
    inputs, against the oracle; L spans several 64-step tiles and ends in a partial one."""
    _check_conv(width, io, dim)


@pytest.mark.parametrize("width", [1, 4, 8])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_conv1d_silu_plain_load_path(width, io, plain_loads):
    """The register-window kernel that serves rows TMA cannot address."""
    _check_conv(width, io, 128)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_conv1d_silu_many_tiles_per_cta(io):
    """More tiles than resident CTAs: every CTA cycles its pipeline stages several times."""
    _check_conv(4, io, 512, batch=4, L=16384, seed=5)


def test_conv1d_then_scan_matches_oracle_chain():
    """The convolution's output fed to the scan as u equals the oracle chain conv -> scan."""
    w_ = WORKLOADS["bf16"].replace(batch=2, L=300, dim=136)
    x = make_inputs(w_, device=DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(7)
    xin = torch.randn(x["u"].shape, generator=g, device=DEV).to(torch.bfloat16)
    wc = torch.randn((w_.dim, 4), generator=g, device=DEV) * 0.5
    bc = torch.randn((w_.dim,), generator=g, device=DEV)
    u = binding.conv1d_silu(xin, wc, bc)
    x["u"] = u
    y, h = binding.fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                       x["delta_bias"])
    assert binding.device_error() == 0
    ur = oracle.conv1d(to_np_io(xin), wc.cpu().numpy(), bc.cpu().numpy(), io="bf16")
    # the scan reads the stored (bf16) u, so the oracle chain uses the library's rounded u only
    # after checking it against the convolution oracle
    assert_within(compare(u, None, ur, None, "bf16"), "bf16", "conv output")
    yr, hr, ym = oracle_full(x)
    assert_within(compare(y, h, yr, hr, "bf16", y_mag=ym), "bf16", "conv -> scan")
