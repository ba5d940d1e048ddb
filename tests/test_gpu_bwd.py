"""GPU parity of the backward pass (sscan_bwd) against the fp64 adjoint oracle: every gradient,
both decay factors, optional operands on and off, ragged sizes, bf16 and fp32 io.

Tolerance (the contract states none for gradients): gradients take the forward's bounds and
metric (parity.py). bf16-typed gradients (du, ddelta, dz of bf16 runs) are compared after
rounding the oracle to bf16, on the survey scale: max 2e-2 and mean 1e-3. fp32-typed gradients
are sums that can cancel (dA adds B*L terms, dB and dC D*N-term sums, du and ddelta N-term
sums of adjoint products): they are compared on the term scale, with each gradient's magnitude
from the oracle (every term by its absolute value), max 1e-4.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from parity import err_stats, round_bf16, to_np_io
from selective_state_space_158_b300 import binding
from selective_state_space_158_b300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TOL_BWD = {"f32": {"max": 1e-4}, "bf16": {"max": 2e-2, "mean": 1e-3}}
IO_GRADS = ("du", "ddelta", "dz")


def _case(io, batch, L, dim, N, euler, opt, seed=3):
    base = WORKLOADS["fp32"] if io == "f32" else WORKLOADS["bf16"]
    w = base.replace(batch=batch, L=L, dim=dim, N=N, has_z=opt, has_D=opt, has_bias=opt)
    x = make_inputs(w, device=DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    dt = x["u"].dtype
    dy = torch.randn(x["u"].shape, generator=g, device=DEV).to(dt)
    dh = torch.randn((batch, dim, N), generator=g, device=DEV)
    h0 = torch.randn((batch, dim, N), generator=g, device=DEV) if opt else None
    softplus = not euler
    if euler:  # keep dt |A| < 2 (see the forward tests)
        x["delta"] = (x["delta"].float().abs() * 0.02).to(dt)
        x["delta_bias"] = None
    return w, x, dy, dh, h0, softplus


def _check(io, batch, L, dim, N, euler, opt, what):
    w, x, dy, dh, h0, softplus = _case(io, batch, L, dim, N, euler, opt)
    got = binding.bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], dy, D=x.get("D"), z=x.get("z"),
                      delta_bias=x.get("delta_bias"), dh_last=dh, softplus=softplus, h0=h0,
                      euler=euler, want_dh0=True)
    torch.cuda.synchronize()
    f = lambda t: None if t is None else t.detach().cpu().numpy()  # noqa: E731
    ref = oracle.bwd(to_np_io(x["u"]), to_np_io(x["delta"]), f(x["A"]), to_np_io(x["B"]),
                     to_np_io(x["C"]), f(x.get("D")),
                     None if x.get("z") is None else to_np_io(x["z"]), f(x.get("delta_bias")),
                     to_np_io(dy), f(dh), softplus=softplus, h0=f(h0), euler=euler, io=w.io)
    mag = oracle.bwd(to_np_io(x["u"]), to_np_io(x["delta"]), f(x["A"]), to_np_io(x["B"]),
                     to_np_io(x["C"]), f(x.get("D")),
                     None if x.get("z") is None else to_np_io(x["z"]), f(x.get("delta_bias")),
                     to_np_io(dy), f(dh), softplus=softplus, h0=f(h0), euler=euler, io=w.io,
                     mag=True)
    ref["dh0"] = ref.get("dh0")
    report = {}
    for k, r in ref.items():
        if r is None:
            continue
        y = got[k].detach().float().cpu().numpy().astype(np.float64)
        io_typed = w.io == "bf16" and k in IO_GRADS
        rr = round_bf16(r) if io_typed else r
        st = err_stats(y, rr) if io_typed else err_stats(y, rr, mag=mag[k])
        report[k] = st
        tol = TOL_BWD[w.io] if k in IO_GRADS else TOL_BWD["f32"]
        assert st["max"] <= tol["max"], f"{what} {k}: max {st['max']:.3g} > {tol['max']}"
        if "mean" in tol:
            assert st["mean"] <= tol["mean"], f"{what} {k}: mean {st['mean']:.3g}"
    print("\nBWD", what, {k: f"{v['max']:.1e}/{v['mean']:.1e}" for k, v in report.items()})


@pytest.mark.parametrize("euler", [False, True])
@pytest.mark.parametrize("opt", [True, False])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_backward(euler, opt, io):
    _check(io, batch=2, L=301, dim=136, N=16, euler=euler, opt=opt,
           what=f"bwd {io} euler={euler} opt={opt}")


@pytest.mark.parametrize("N,dim,L", [(5, 37, 64), (1, 40, 17), (8, 200, 33)])
def test_backward_small_state_and_ragged(N, dim, L):
    _check("f32", batch=3, L=L, dim=dim, N=N, euler=False, opt=True, what=f"bwd N={N} dim={dim}")


def test_backward_is_deterministic():
    w, x, dy, dh, h0, softplus = _case("bf16", 2, 200, 136, 16, False, True)
    run = lambda: binding.bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], dy, D=x["D"],  # noqa
                              z=x["z"], delta_bias=x["delta_bias"], dh_last=dh, h0=h0,
                              want_dh0=True)
    a, b = run(), run()
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("io,N,dim,batch", [("bf16", 16, 4096, 4), ("f32", 5, 3000, 5)])
def test_backward_many_tiles(io, N, dim, batch):
    """More (batch row, channel group) tiles than three CTAs per SM hold: the kernel built for
    four resident CTAs, on the staged path (bf16, N 16) and the register path (N 5)."""
    _check(io, batch=batch, L=21, dim=dim, N=N, euler=False, opt=True,
           what=f"bwd many tiles {io} N={N}")


def _misaligned(t):
    """A contiguous copy of t whose data starts one element past a 16-byte boundary."""
    flat = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
    out = flat[1:].view(t.shape)
    out.copy_(t)
    return out


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_backward_unaligned_inputs(io):
    """Inputs that do not start on a 16-byte boundary take the register-load path and give the
    same gradients as aligned ones."""
    w, x, dy, dh, h0, softplus = _case(io, 2, 77, 136, 16, False, True)
    run = lambda xx, dd: binding.bwd(xx["u"], xx["delta"], xx["A"], xx["B"], xx["C"], dd,  # noqa
                                     D=xx["D"], z=xx["z"], delta_bias=xx["delta_bias"],
                                     dh_last=dh, h0=h0, want_dh0=True)
    ref = run(x, dy)
    xm = dict(x)
    for k in ("u", "delta", "z", "B", "C"):
        xm[k] = _misaligned(x[k])
    got = run(xm, _misaligned(dy))
    torch.cuda.synchronize()
    for k in ref:
        r, gq = ref[k].float(), got[k].float()
        tol = 1e-5 if (io == "f32" or k not in IO_GRADS) else 1e-2
        err = ((gq - r).abs().max() / r.abs().max().clamp_min(1e-30)).item()
        assert err <= tol, f"{k}: {err:.3g}"


@pytest.mark.parametrize("segments", [2, 3, 7])
@pytest.mark.parametrize("euler", [False, True])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_backward_time_segments(segments, euler, io, tune):
    """The sequence split into time segments: an aggregate pass carries the adjoint of every
    later segment back to each segment's end (zero-order hold and first-order factors)."""
    tune(bwd_segments=segments)
    _check(io, batch=2, L=301 if segments != 7 else 1777, dim=136, N=16, euler=euler, opt=True,
           what=f"bwd segments={segments} {io} euler={euler}")


def test_backward_time_segments_register_path(tune):
    """Time segments on the register-load path (N 5) with a ragged last segment."""
    tune(bwd_segments=4)
    _check("f32", batch=3, L=250, dim=37, N=5, euler=False, opt=True, what="bwd segments N=5")
