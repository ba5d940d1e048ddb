"""Shared parity helpers: the error metric, bf16 rounding of oracle values and oracle calls on
torch inputs.

Error metric. The tolerances' "relative error" is undefined near zero, so every compared value i
is measured against a floor:

    err_i = |y_i - r_i| / max(|r_i|, FLOOR * s_i),   FLOOR = 1e-2

with r the oracle (rounded to bf16 first when the library's output is bf16, because rounding
alone would otherwise contribute ~1.4e-3 mean relative error) and s_i one of two scales:

* survey scale, s_i = rms(r) over the compared set: reported for every comparison, and the one
  asserted for bf16 outputs and for the fp32 final state h_last;
* term scale, s_i = max(rms(r), m_i), m_i the magnitude of value i's terms (the oracle's sum of
  their absolute values: every state, readout, skip and gate term, or every term of a gradient):
  asserted for fp32-typed outputs that are sums which can cancel (y of fp32 io, gradients).

Why the term scale for fp32 sums. The method prescribes fp32 state and fp32 accumulation. An
output y_t = (sum_n C_t[n] h_t[n] + D u_t) SiLU(z_t) computed in fp32 carries a rounding error
of order 2^-24 m_i however it is evaluated, and where the terms cancel (|y_i| far below m_i)
that error, measured against 1e-2 rms(r), exceeds 1e-4: a correctly rounded fp32 evaluation of
the full fp32 workload (every operation rounded exactly once) reaches about 1.4e-4 on the survey
scale (tests/test_fp32_evaluation_bound.py reproduces it on one batch row) and about 4e-5 on the
term scale. The term scale keeps the survey's floor constant and its rms for every output whose
terms do not cancel; it still fails an evaluation whose error compounds (per-step SFU
exponentials without re-anchoring: 1.7e-4 on the term scale) and any wrong index, sign or term.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

FLOOR = 1e-2
TOL = {"f32": {"max": 1e-4}, "bf16": {"max": 2e-2, "mean": 1e-3}}


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), returned as float64.
    Exact for normal-range values: keeps 8 significant bits of the float64 mantissa."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)  # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def err_stats(y: np.ndarray, r: np.ndarray, floor: float = FLOOR, mag=None) -> dict:
    """max / mean of err_i (survey scale, or term scale when the magnitudes ``mag`` are given)
    and the normwise max|y - r| / max|r|."""
    y = np.asarray(y, dtype=np.float64).ravel()
    r = np.asarray(r, dtype=np.float64).ravel()
    if r.size == 0:
        return {"max": 0.0, "mean": 0.0, "normwise": 0.0, "n": 0}
    rms = float(np.sqrt(np.mean(r * r)))
    scale = rms if mag is None else np.maximum(rms, np.asarray(mag, dtype=np.float64).ravel())
    denom = np.maximum(np.abs(r), floor * scale)
    denom = np.where(denom == 0, 1.0, denom)
    e = np.abs(y - r) / denom
    nw = float(np.abs(y - r).max() / max(np.abs(r).max(), 1e-300))
    if not np.all(np.isfinite(y)):
        return {"max": float("inf"), "mean": float("inf"), "normwise": float("inf"), "n": r.size}
    return {"max": float(e.max()), "mean": float(e.mean()), "normwise": nw, "n": int(r.size)}


def to_np_io(t: torch.Tensor) -> np.ndarray:
    """A CPU copy in the oracle's io form: float32 values or bf16 bit patterns (uint16)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    raise TypeError(t.dtype)


def io_name(t: torch.Tensor) -> str:
    return "f32" if t.dtype == torch.float32 else "bf16"


def oracle_full(x: dict, softplus: bool = True, h0=None, euler: bool = False):
    """Oracle on whole tensors; h0 a float32 torch tensor or None. Returns (y, h_last, mag)."""
    io = io_name(x["u"])
    g = lambda k: None if x.get(k) is None else to_np_io(x[k])  # noqa: E731
    f = lambda k: None if x.get(k) is None else x[k].detach().cpu().numpy()  # noqa: E731
    return oracle.fwd(g("u"), g("delta"), f("A"), g("B"), g("C"), f("D"), g("z"),
                      f("delta_bias"), softplus=softplus, io=io,
                      h0=None if h0 is None else h0.detach().cpu().numpy(), euler=euler,
                      want_mag=True)


def compare(y_gpu: torch.Tensor, h_gpu, y_ref: np.ndarray, h_ref, io: str, y_mag=None) -> dict:
    """Error stats of y (against the bf16-rounded oracle for bf16 io) and h_last (fp32, never
    rounded): {'y': survey scale, 'y_term': term scale (when y_mag is given), 'y_unrounded':
    survey scale against the unrounded oracle, 'h': survey scale}."""
    yg = y_gpu.detach().float().cpu().numpy().astype(np.float64)
    r = round_bf16(y_ref) if io == "bf16" else y_ref
    res = {"y": err_stats(yg, r), "y_unrounded": err_stats(yg, y_ref)}
    if y_mag is not None:
        res["y_term"] = err_stats(yg, r, mag=y_mag)
    if h_gpu is not None:
        res["h"] = err_stats(h_gpu.detach().cpu().numpy().astype(np.float64), h_ref)
    return res


def assert_within(res: dict, io: str, what: str = ""):
    """bf16 io: y on the survey scale (max and mean). fp32 io: y on the term scale when it was
    computed, else the survey scale. h_last: survey scale, with the io's max bound."""
    tol = TOL[io]
    ykey = "y_term" if (io == "f32" and "y_term" in res) else "y"
    for key in (ykey, "h"):
        if key not in res:
            continue
        st = res[key]
        assert st["max"] <= tol["max"], f"{what} {key}: max rel err {st['max']:.3g} > {tol['max']}"
        if "mean" in tol and key == "y":
            assert st["mean"] <= tol["mean"], \
                f"{what} {key}: mean rel err {st['mean']:.3g} > {tol['mean']}"
