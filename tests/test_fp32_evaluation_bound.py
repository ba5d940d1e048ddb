"""What fp32 arithmetic itself can reach on the fp32 workload, under both scales of the parity
metric (parity.py): a host evaluation of one batch row of the fp32 workload (batch row of
8 x 2048 x 1536, N 16, gate and skip on) in which every operation is rounded exactly once to
fp32 (decay factors, steps, inputs, state, readout in the order the four-lane kernel sums it),
compared with the fp64 oracle.

This is the evidence for the term scale: the best possible fp32 evaluation of the method
exceeds the survey scale's 1e-4 on outputs whose terms cancel, while it sits well inside 1e-4
on the term scale. CPU only, about ten seconds.
"""
import numpy as np

import oracle
from parity import err_stats
from selective_state_space_158_b300.inputs import WORKLOADS, make_inputs

F32, F64 = np.float32, np.float64


def _fma(a, b, c):
    """fp32 fused multiply-add (exact product and sum in float64, one rounding to fp32)."""
    return (a.astype(F64) * b.astype(F64) + c.astype(F64)).astype(F32)


def _rounded_fp32_scan(u, dl, z, B, C, A, D, bias):
    L, dim = u.shape
    N = A.shape[1]
    x = (dl + bias[None, :]).astype(F32)
    x64 = x.astype(F64)
    dt = np.where(x64 > 0, x64 + np.log1p(np.exp(-x64)), np.log1p(np.exp(x64))).astype(F32)
    dtu = (dt * u).astype(F32)
    sil = (z.astype(F64) / (1 + np.exp(-z.astype(F64)))).astype(F32)
    h = np.zeros((dim, N), F32)
    y = np.zeros((L, dim), F32)
    for t in range(L):
        a = np.exp(dt[t].astype(F64)[:, None] * A.astype(F64)).astype(F32)
        b = (dtu[t][:, None] * B[t][None, :]).astype(F32)
        h = _fma(a, h, b)
        c = np.broadcast_to(C[t][None, :], (dim, N))
        part = []
        for g in range(N // 4):  # four lanes of four states: (n0, n0+2), (n0+1, n0+3), then pairs
            n0 = 4 * g
            ax = _fma(c[:, n0 + 2], h[:, n0 + 2], (c[:, n0] * h[:, n0]).astype(F32))
            ay = _fma(c[:, n0 + 3], h[:, n0 + 3], (c[:, n0 + 1] * h[:, n0 + 1]).astype(F32))
            part.append((ax + ay).astype(F32))
        acc = ((part[0] + part[2]).astype(F32) + (part[1] + part[3]).astype(F32)).astype(F32)
        y[t] = (_fma(D, u[t], acc) * sil[t]).astype(F32)
    return y


def test_correctly_rounded_fp32_evaluation_on_both_scales():
    w = WORKLOADS["fp32"].replace(batch=1)
    x = make_inputs(w, device="cpu")
    f = {k: v.numpy() for k, v in x.items()}
    y = _rounded_fp32_scan(f["u"][0], f["delta"][0], f["z"][0], f["B"][0], f["C"][0], f["A"],
                           f["D"], f["delta_bias"])
    r, _, mag = oracle.fwd(f["u"], f["delta"], f["A"], f["B"], f["C"], f["D"], f["z"],
                           f["delta_bias"], want_mag=True)
    survey = err_stats(y, r[0])
    term = err_stats(y, r[0], mag=mag[0])
    print(f"correctly rounded fp32: survey scale max {survey['max']:.3g}, "
          f"term scale max {term['max']:.3g}")
    assert survey["max"] > 1e-4  # the survey scale alone is out of fp32's reach here
    assert term["max"] < 6e-5 and term["max"] < 0.5 * survey["max"]
