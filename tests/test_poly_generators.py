"""The polynomial constants in the kernels' device header are the ones their committed generator
scripts produce, and those polynomials meet their stated accuracy (CPU, fp32 emulation)."""
import os
import re
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "selective_state_space_158_b300", "csrc")
sys.path.insert(0, CSRC)

import gen_exp2_poly  # noqa: E402
import gen_softplus_poly  # noqa: E402


def _header_arrays():
    text = open(os.path.join(CSRC, "sscan_device.cuh")).read()
    arrays = re.findall(r"constexpr float c\[(\d+)\] = \{([^}]*)\}", text)
    return [np.array([float(v.strip().rstrip("f")) for v in body.split(",")], dtype=np.float32)
            for _, body in arrays]


def test_exp2_constants_match_generator_and_accuracy():
    cf = gen_exp2_poly.coefficients()
    assert any(a.shape == cf.shape and np.array_equal(a, cf) for a in _header_arrays())
    mx, mean = gen_exp2_poly.errors(cf)
    assert mx <= 1.1e-7 and abs(mean) <= 1e-8


def test_softplus_constants_match_generator_and_accuracy():
    cf = gen_softplus_poly.coefficients()
    assert any(a.shape == cf.shape and np.array_equal(a, cf) for a in _header_arrays())
    assert gen_softplus_poly.max_rel_error(cf) <= 2e-7
    cf6 = gen_softplus_poly.coefficients(6)  # the bf16 io path's shorter polynomial
    assert any(a.shape == cf6.shape and np.array_equal(a, cf6) for a in _header_arrays())
    assert gen_softplus_poly.max_rel_error(cf6) <= 2e-6
