"""Seeded random shapes through the automatic kernel choice (lane kernel in its layouts and CTA
sizes, time segments, the time-lane kernel, the plain-load fallback for unaligned shapes),
each against the fp64 oracle over whole tensors: batch 1-5, L 1-9000, D 1-400, N 1-16, fp32 or
bf16, every optional operand on or off, softplus on or off, an initial state or none."""
import numpy as np
import pytest
import torch

from parity import assert_within, compare, oracle_full
from selective_state_space_158_b300 import binding
from selective_state_space_158_b300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    io = "f32" if rng.random() < 0.5 else "bf16"
    base = WORKLOADS["fp32"] if io == "f32" else WORKLOADS["bf16"]
    batch = int(rng.integers(1, 6))
    L = int(rng.choice([1, 7, 100, 257, 1000, 4097, 9000]))
    dim = int(rng.choice([1, 8, 24, 64, 136, 200, 400]))
    N = int(rng.choice([1, 5, 16, 16]))
    w = base.replace(batch=batch, L=L, dim=dim, N=N, seed_index=10 + seed)
    opts = {"D": rng.random() < 0.7, "z": rng.random() < 0.7, "bias": rng.random() < 0.8,
            "softplus": rng.random() < 0.8, "h0": rng.random() < 0.3}
    return w, opts


@pytest.mark.parametrize("seed", range(24))
def test_random_shape_against_oracle(seed):
    w, o = _case(seed)
    x = make_inputs(w, device=DEV)
    if not o["D"]:
        x["D"] = None
    if not o["z"]:
        x["z"] = None
    if not o["bias"]:
        x["delta_bias"] = None
    if not o["softplus"]:  # positive steps as given
        x["delta"] = (x["delta"].float().abs() * 0.05).to(x["u"].dtype)
        x["delta_bias"] = None
    h0 = None
    if o["h0"]:
        g = torch.Generator(device=DEV)
        g.manual_seed(seed)
        h0 = torch.randn((w.batch, w.dim, w.N), generator=g, device=DEV, dtype=torch.float32)
    y, h = binding.fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x.get("D"), x.get("z"),
                       x.get("delta_bias"), softplus=o["softplus"], h0=h0)
    assert binding.device_error() == 0
    yr, hr, ym = oracle_full(x, o["softplus"], h0=h0)
    what = f"seed {seed}: {w.io} b{w.batch} L{w.L} D{w.dim} N{w.N} {o}"
    assert_within(compare(y, h, yr, hr, w.io, y_mag=ym), w.io, what)
