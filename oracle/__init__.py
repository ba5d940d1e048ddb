"""fp64 CPU oracle of the S6 selective-scan forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import this package. The product library never loads it: the CUDA
path and this oracle share no code (no kernels, headers, helpers, tables or constants).

The arithmetic lives in ``sscan_oracle.c`` (plain sequential loops in double precision, one
POSIX thread per group of independent channels); this module compiles it with gcc and marshals
numpy arrays to it. See the C file's header for what is computed and which page and section each
step follows.

Every function here has at least one pin in ``tests/test_oracle_pins.py`` against values the
pages fix (the worked LTI demo of "架构变体：Mamba/SSM"), closed forms (causal convolution,
the semiseparable-matrix form), invariants (Delta -> 0, associativity of the scan operator)
and library routines (``numpy.logaddexp``, ``scipy.special.expit``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sscan_oracle.c")
_LIB = os.path.join(_HERE, "libsscan_oracle.so")

_lib_cache: dict = {}


def build(mutant: int = 0, out: Optional[str] = None) -> str:
    """Compile the C oracle with gcc (no fast-math: IEEE double semantics) and return its path.

    ``mutant`` != 0 builds a deliberately broken copy; the pin tests use those copies to show
    that each plausible mistake is caught by at least one pin.
    """
    if out is None:
        out = _LIB if mutant == 0 else os.path.join(_HERE, f"libsscan_oracle_m{mutant}.so")
    if mutant == 0 and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           f"-DSSCAN_ORACLE_MUTANT={int(mutant)}", "-o", out, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle shared library."""
    path = path or build()
    if path in _lib_cache:
        return _lib_cache[path]
    lib = ctypes.CDLL(path)
    i64, vp, dp, fp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int
    lib.sscan_oracle_fwd.argtypes = [vp, vp, fp, vp, vp, fp, vp, fp, ci, dp, dp, dp,
                                     i64, i64, i64, i64, ci, ci]
    lib.sscan_oracle_fwd.restype = ci
    lib.sscan_oracle_channel.argtypes = [vp, vp, vp, i64, fp, vp, vp, fp, fp, ci,
                                         i64, i64, ci, dp, i64, dp, dp]
    lib.sscan_oracle_channel.restype = None
    lib.sscan_oracle_fwd_ex.argtypes = [vp, vp, fp, vp, vp, fp, vp, fp, ci, fp, ci, dp, dp, dp,
                                        i64, i64, i64, i64, ci, ci]
    lib.sscan_oracle_fwd_ex.restype = ci
    lib.sscan_oracle_channel_ex.argtypes = [vp, vp, vp, i64, fp, vp, vp, fp, fp, ci, fp, ci,
                                            i64, i64, ci, dp, i64, dp, dp]
    lib.sscan_oracle_channel_ex.restype = None
    lib.sscan_oracle_conv1d.argtypes = [vp, fp, fp, vp, ci, dp, i64, i64, i64, i64, ci]
    lib.sscan_oracle_conv1d.restype = ci
    lib.sscan_oracle_bwd.argtypes = [vp, vp, fp, vp, vp, fp, vp, fp, ci, fp, ci, vp, fp,
                                     dp, dp, dp, dp, dp, dp, dp, dp, dp, i64, i64, i64, i64, ci,
                                     ci]
    lib.sscan_oracle_bwd.restype = ci
    _lib_cache[path] = lib
    return lib


def _io_array(a: np.ndarray, io: str) -> np.ndarray:
    if io == "f32":
        if a.dtype != np.float32:
            raise TypeError(f"f32 io expects float32 arrays, got {a.dtype}")
    elif io == "bf16":
        if a.dtype != np.uint16:
            raise TypeError(f"bf16 io expects the uint16 bit patterns, got {a.dtype}")
    else:
        raise ValueError(io)
    return np.ascontiguousarray(a)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def fwd(u, delta, A, B, C, Dskip=None, z=None, delta_bias=None, softplus: bool = True,
        io: str = "f32", threads: Optional[int] = None, want_mag: bool = False, lib=None,
        h0=None, euler: bool = False):
    """Selective-scan forward over whole tensors.

    u, delta, z: (batch, L, dim); B, C: (batch, L, N); A: (dim, N) float32; Dskip, delta_bias:
    (dim,) float32; h0: (batch, dim, N) float32 initial state or None for zero; ``euler``
    selects the first-order factor ``1 + dt A`` instead of ``exp(dt A)``. For ``io="bf16"`` the
    io tensors are uint16 arrays holding bf16 bit patterns.
    Returns ``(y, h_last)`` as float64 arrays of shapes (batch, L, dim) and (batch, dim, N), plus
    the absolute-value magnitude of every output when ``want_mag``.
    """
    lib = lib or load()
    u, delta = _io_array(u, io), _io_array(delta, io)
    B, C = _io_array(B, io), _io_array(C, io)
    z = None if z is None else _io_array(z, io)
    batch, L, dim = u.shape
    N = B.shape[2]
    assert delta.shape == u.shape and B.shape == C.shape == (batch, L, N)
    assert z is None or z.shape == u.shape
    A = np.ascontiguousarray(A, dtype=np.float32)
    assert A.shape == (dim, N)
    Dskip = None if Dskip is None else np.ascontiguousarray(Dskip, dtype=np.float32)
    delta_bias = None if delta_bias is None else np.ascontiguousarray(delta_bias, dtype=np.float32)
    if h0 is not None:
        if h0.dtype != np.float32 or h0.shape != (batch, dim, N):
            raise TypeError(f"h0 must be float32 of shape {(batch, dim, N)}")
        h0 = np.ascontiguousarray(h0)
    y = np.empty((batch, L, dim), dtype=np.float64)
    h = np.empty((batch, dim, N), dtype=np.float64)
    mag = np.empty_like(y) if want_mag else None
    nt = threads or os.cpu_count() or 1
    rc = lib.sscan_oracle_fwd_ex(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(Dskip),
                                 _ptr(z), _ptr(delta_bias), int(bool(softplus)), _ptr(h0),
                                 int(bool(euler)), _ptr(y), _ptr(h), _ptr(mag), batch, L, dim, N,
                                 int(io == "bf16"), int(nt))
    if rc != 0:
        raise ValueError("oracle rejected the sizes")
    return (y, h, mag) if want_mag else (y, h)


def fwd_channel(u, delta, A_d, B, C, Dskip_d=None, z=None, bias_d=None, softplus: bool = True,
                io: str = "f32", want_mag: bool = False, lib=None, h0_d=None,
                euler: bool = False):
    """One channel: u, delta, z are (L,) io arrays, B and C (L, N), A_d (N,) float32, Dskip_d and
    bias_d Python floats (stored as float32) or None, h0_d (N,) float32 or None. Returns
    ``(y (L,), h_last (N,))`` in float64 (plus the magnitude when ``want_mag``). Used to check
    sampled channels of large runs."""
    lib = lib or load()
    u, delta = _io_array(u, io), _io_array(delta, io)
    B, C = _io_array(B, io), _io_array(C, io)
    z = None if z is None else _io_array(z, io)
    L = u.shape[0]
    N = B.shape[1]
    A_d = np.ascontiguousarray(A_d, dtype=np.float32)
    Dv = None if Dskip_d is None else np.array([Dskip_d], dtype=np.float32)
    bv = None if bias_d is None else np.array([bias_d], dtype=np.float32)
    y = np.empty(L, dtype=np.float64)
    h = np.empty(N, dtype=np.float64)
    mag = np.empty(L, dtype=np.float64) if want_mag else None
    h0v = None if h0_d is None else np.ascontiguousarray(h0_d, dtype=np.float32)
    lib.sscan_oracle_channel_ex(_ptr(u), _ptr(delta), _ptr(z), 1, _ptr(A_d), _ptr(B), _ptr(C),
                                _ptr(Dv), _ptr(bv), int(bool(softplus)), _ptr(h0v),
                                int(bool(euler)), L, N, int(io == "bf16"), _ptr(y), 1, _ptr(h),
                                _ptr(mag))
    return (y, h, mag) if want_mag else (y, h)


def conv1d(x, w, bias=None, x_prev=None, silu: bool = True, io: str = "f32", lib=None):
    """Causal depthwise convolution over time, then SiLU (see ``sscan_oracle_conv1d``).

    x: (batch, L, dim) io array; w: (dim, width) float32; bias: (dim,) float32 or None; x_prev:
    (batch, width - 1, dim) io array or None (zeros before t = 0). Returns y (batch, L, dim)
    float64.
    """
    lib = lib or load()
    x = _io_array(x, io)
    batch, L, dim = x.shape
    w = np.ascontiguousarray(w, dtype=np.float32)
    assert w.shape[0] == dim
    width = w.shape[1]
    bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    if x_prev is not None:
        x_prev = _io_array(x_prev, io)
        assert x_prev.shape == (batch, width - 1, dim)
    y = np.empty((batch, L, dim), dtype=np.float64)
    rc = lib.sscan_oracle_conv1d(_ptr(x), _ptr(w), _ptr(bias), _ptr(x_prev), int(bool(silu)),
                                 _ptr(y), batch, L, dim, width, int(io == "bf16"))
    if rc != 0:
        raise ValueError("oracle rejected the sizes")
    return y


def bwd(u, delta, A, B, C, Dskip, z, delta_bias, dy, dh_last=None, softplus: bool = True,
        h0=None, euler: bool = False, io: str = "f32", lib=None, mag: bool = False):
    """Gradients of sum(dy * y) + sum(dh_last * h_last) for the forward of ``fwd`` (see
    ``sscan_oracle_bwd``). dy: (batch, L, dim) io array; dh_last: (batch, dim, N) float32 or
    None. Returns a dict of float64 arrays: du, ddelta, dA, dB, dC, and dz / dD / ddelta_bias /
    dh0 when z / Dskip / delta_bias / h0 are given. With ``mag`` the same dict holds each
    gradient's magnitude (every term taken by its absolute value) instead."""
    lib = lib or load()
    u, delta, dy = _io_array(u, io), _io_array(delta, io), _io_array(dy, io)
    B, C = _io_array(B, io), _io_array(C, io)
    z = None if z is None else _io_array(z, io)
    batch, L, dim = u.shape
    N = B.shape[2]
    A = np.ascontiguousarray(A, dtype=np.float32)
    Dskip = None if Dskip is None else np.ascontiguousarray(Dskip, dtype=np.float32)
    delta_bias = None if delta_bias is None else np.ascontiguousarray(delta_bias, dtype=np.float32)
    h0 = None if h0 is None else np.ascontiguousarray(h0, dtype=np.float32)
    dh_last = None if dh_last is None else np.ascontiguousarray(dh_last, dtype=np.float32)
    out = {"du": np.empty((batch, L, dim)), "ddelta": np.empty((batch, L, dim)),
           "dA": np.empty((dim, N)), "dB": np.empty((batch, L, N)), "dC": np.empty((batch, L, N))}
    out["dz"] = np.empty((batch, L, dim)) if z is not None else None
    out["dD"] = np.empty(dim) if Dskip is not None else None
    out["ddelta_bias"] = np.empty(dim) if delta_bias is not None else None
    out["dh0"] = np.empty((batch, dim, N)) if h0 is not None else None
    rc = lib.sscan_oracle_bwd(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(Dskip),
                              _ptr(z), _ptr(delta_bias), int(bool(softplus)), _ptr(h0),
                              int(bool(euler)), _ptr(dy), _ptr(dh_last), _ptr(out["du"]),
                              _ptr(out["ddelta"]), _ptr(out["dA"]), _ptr(out["dB"]),
                              _ptr(out["dC"]), _ptr(out["dD"]), _ptr(out["dz"]),
                              _ptr(out["ddelta_bias"]), _ptr(out["dh0"]), batch, L, dim, N,
                              int(io == "bf16"), int(bool(mag)))
    if rc != 0:
        raise ValueError("oracle rejected the sizes")
    return {k: v for k, v in out.items() if v is not None}
