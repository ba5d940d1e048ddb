"""Shared parity helpers: the error metric, bf16 rounding of oracle values, oracle calls on
torch inputs, and sampled-channel checks for workloads too large for a whole-tensor oracle run.

Error metric (the tolerance's "relative error", which the task leaves undefined near zero):
    err_i = |y_i - r_i| / max(|r_i|, FLOOR * rms(r))
with r the oracle (rounded to bf16 first when the library's output is bf16, because rounding
alone would otherwise contribute ~1.4e-3 mean relative error) and rms over the compared set.

FLOOR = 0.1: the per-step decay factor exp(dt A) is rounded to fp32 (and the SFU exponential
is accurate to ~2 ulp), and that error compounds over the state's memory of about
1 / (dt |A|) steps; for the slowest fp32 workload channels (dt = 1e-3, A = -1) this bounds the
state's relative error near 1e-4 and the readout's absolute error near 1e-5 rms(y). The floor
keeps near-zero outputs from turning that absolute error into an unbounded relative one; a
wrong index, sign or term still produces O(1) errors under this metric.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

FLOOR = 0.1
TOL = {"f32": {"max": 1e-4}, "bf16": {"max": 2e-2, "mean": 1e-3}}


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), returned as float64.
    Exact for normal-range values: keeps 8 significant bits of the float64 mantissa."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)  # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def err_stats(y: np.ndarray, r: np.ndarray, floor: float = FLOOR) -> dict:
    y = np.asarray(y, dtype=np.float64).ravel()
    r = np.asarray(r, dtype=np.float64).ravel()
    if r.size == 0:
        return {"max": 0.0, "mean": 0.0, "normwise": 0.0, "n": 0}
    rms = float(np.sqrt(np.mean(r * r)))
    denom = np.maximum(np.abs(r), floor * rms)
    denom[denom == 0] = 1.0
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
    """Oracle on whole tensors (small workloads); h0 a float32 torch tensor or None."""
    io = io_name(x["u"])
    g = lambda k: None if x.get(k) is None else to_np_io(x[k])  # noqa: E731
    f = lambda k: None if x.get(k) is None else x[k].detach().cpu().numpy()  # noqa: E731
    return oracle.fwd(g("u"), g("delta"), f("A"), g("B"), g("C"), f("D"), g("z"),
                      f("delta_bias"), softplus=softplus, io=io,
                      h0=None if h0 is None else h0.detach().cpu().numpy(), euler=euler)


def oracle_channels(x: dict, chans, softplus: bool = True):
    """Oracle on selected (b, d) channels only; reads back just those slices."""
    io = io_name(x["u"])
    out = []
    for b, d in chans:
        sl = lambda k: None if x.get(k) is None else to_np_io(x[k][b, :, d])  # noqa: E731
        y, h = oracle.fwd_channel(
            sl("u"), sl("delta"), x["A"][d].cpu().numpy(), to_np_io(x["B"][b]),
            to_np_io(x["C"][b]),
            None if x.get("D") is None else float(x["D"][d]), sl("z"),
            None if x.get("delta_bias") is None else float(x["delta_bias"][d]),
            softplus=softplus, io=io)
        out.append((y, h))
    return out


def compare(y_gpu: torch.Tensor, h_gpu, y_ref: np.ndarray, h_ref, io: str) -> dict:
    """Error stats of y (against the bf16-rounded oracle for bf16 io) and h_last (fp32, never
    rounded). Returns {'y': stats, 'y_unrounded': stats, 'h': stats}."""
    yg = y_gpu.detach().float().cpu().numpy().astype(np.float64)
    r = round_bf16(y_ref) if io == "bf16" else y_ref
    res = {"y": err_stats(yg, r), "y_unrounded": err_stats(yg, y_ref)}
    if h_gpu is not None:
        res["h"] = err_stats(h_gpu.detach().cpu().numpy().astype(np.float64), h_ref)
    return res


def assert_within(res: dict, io: str, what: str = ""):
    tol = TOL[io]
    for key in ("y", "h"):
        if key not in res:
            continue
        st = res[key]
        assert st["max"] <= tol["max"], f"{what} {key}: max rel err {st['max']:.3g} > {tol['max']}"
        if "mean" in tol:
            assert st["mean"] <= tol["mean"], \
                f"{what} {key}: mean rel err {st['mean']:.3g} > {tol['mean']}"
