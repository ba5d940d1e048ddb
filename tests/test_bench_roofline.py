"""The bench's roofline arithmetic on synthetic probe rates (no GPU): the compute peak is the
slower pipe for one update (one ex2, four FP32 operations), the binding bound is the slower of
HBM and compute, frac = achieved / peak, and the step-loop fraction uses the loop probe."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from selective_state_space_158_b300.inputs import WORKLOADS  # noqa: E402


def _rates(ex2=32.0, ffma=123.0, ffma2=109.0, loop=20.0):
    r = {"ex2": {"ex2_per_clk_sm": ex2, "fp32_per_clk_sm": 0.0},
         "ffma": {"ex2_per_clk_sm": 0.0, "fp32_per_clk_sm": ffma},
         "ffma2": {"ex2_per_clk_sm": 0.0, "fp32_per_clk_sm": ffma2},
         "mix_packed": {"ex2_per_clk_sm": 20.6, "fp32_per_clk_sm": 82.4},
         "mix_scalar": {"ex2_per_clk_sm": 21.4, "fp32_per_clk_sm": 85.6},
         "step_loop": {"states16_readout_warps24": loop}}
    return r


def test_compute_peak_is_the_slower_pipe():
    pk = bench.update_peak(_rates(), 148, 2000.0)
    assert pk["updates_per_clk_sm"] == pytest.approx(min(32.0, 123.0 / 4))
    assert pk["binding_pipe"] == "FP32"
    assert pk["updates_per_s"] == pytest.approx(123.0 / 4 * 148 * 2000e6)
    pk = bench.update_peak(_rates(ex2=16.0), 148, 2000.0)
    assert pk["binding_pipe"] == "SFU" and pk["updates_per_clk_sm"] == 16.0


@pytest.mark.parametrize("key", ["fp32", "long"])
def test_roofline_bound_and_fractions(key):
    w = WORKLOADS[key]
    pk = bench.update_peak(_rates(), 148, 2000.0)
    hbm = 6500.0
    t_hbm = w.io_bytes() / (hbm * 1e9)
    t_alu = w.elems / pk["updates_per_s"]
    sec = 2.5 * max(t_hbm, t_alu)  # a launch 2.5x slower than its binding roofline
    roof = bench.scan_roofline(w, sec, pk, hbm, "test", None)
    assert roof["bound"] == ("hbm" if t_hbm >= t_alu else "alu")
    assert roof["frac"] == pytest.approx(1 / 2.5)
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
    assert roof["hbm_frac"] == pytest.approx(t_hbm / sec)
    assert roof["alu_frac"] == pytest.approx(t_alu / sec)
    loop_ups = 20.0 * 148 * 2000e6
    assert roof["step_loop_frac"] == pytest.approx(w.elems / sec / loop_ups)
    assert roof["traffic"] is None
