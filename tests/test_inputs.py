"""Host-side checks of the seeded input recipe (no GPU)."""
import math

import numpy as np
import torch

from selective_state_space_158_b300.inputs import WORKLOADS, make_inputs


def test_deterministic_and_independent_per_tensor():
    w = WORKLOADS["tiny"]
    a = make_inputs(w)
    b = make_inputs(w)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    c = make_inputs(w, seed=123)
    assert not torch.equal(a["u"], c["u"])
    # a tensor does not depend on which other tensors are present
    d = make_inputs(w.replace(has_z=True))
    assert torch.equal(a["u"], d["u"]) and torch.equal(a["B"], d["B"])


def test_shapes_dtypes_and_step_range():
    for key in ("tiny",):
        w = WORKLOADS[key]
        x = make_inputs(w)
        assert x["u"].shape == (w.batch, w.L, w.dim) and x["u"].dtype == torch.float32
        assert x["B"].shape == (w.batch, w.L, w.N) and x["C"].shape == x["B"].shape
        assert x["A"].shape == (w.dim, w.N) and x["A"].dtype == torch.float32
        assert torch.equal(x["A"][3], -torch.arange(1, w.N + 1, dtype=torch.float32))
        # softplus(bias) lands in the workload's step range
        dt0 = np.logaddexp(0.0, x["delta_bias"].double().numpy())
        lo, hi = w.dt_range
        assert dt0.min() >= lo * (1 - 1e-5) and dt0.max() <= hi * (1 + 1e-5)
        assert abs(float(x["u"].mean())) < 0.05 and abs(float(x["u"].std()) - 1) < 0.05


def test_bf16_workload_rounding_and_A_pattern():
    w = WORKLOADS["bf16"].replace(batch=1, L=64, dim=128)
    x = make_inputs(w)
    assert x["u"].dtype == torch.bfloat16 and x["A"].dtype == torch.float32
    a = -x["A"].double().numpy()
    assert a.min() >= 1.0 - 1e-6 and a.max() <= 16.0 + 1e-5
    assert len(np.unique(a)) > 1000  # drawn per (d, n)


def test_io_bytes_matches_hand_count():
    w = WORKLOADS["fp32"]
    bld, bln = 8 * 2048 * 1536, 8 * 2048 * 16
    expect = 4 * (3 * bld + 2 * bln) + 1536 * 16 * 4 + 2 * 1536 * 4 + 4 * bld + 8 * 1536 * 16 * 4
    assert w.io_bytes() == expect
    assert w.elems == 8 * 2048 * 1536 * 16
    assert math.isclose(WORKLOADS["long"].elems, 2.58e10, rel_tol=0.01)
