"""Thin ctypes binding of libsscan: argument marshalling only.

Every step of the scan runs in the library's CUDA kernels; this module only checks tensor
properties, passes ``data_ptr()`` values and the current CUDA stream to the C entry points, and
turns status codes into exceptions. There is no fallback: if ``libsscan.so`` is missing or no
CUDA device is present, the calls raise.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsscan.so")

SSCAN_F32, SSCAN_BF16 = 0, 1
SSCAN_DISC_ZOH, SSCAN_DISC_EULER = 0, 1
STATUS = {0: "SSCAN_OK", 1: "SSCAN_ERR_INVALID_ARG", 2: "SSCAN_ERR_UNSUPPORTED",
          3: "SSCAN_ERR_CUDA", 4: "SSCAN_ERR_CARRY_TIMEOUT", 5: "SSCAN_ERR_SCRATCH_TOO_SMALL"}

# Every symbol include/sscan.h declares, with its ctypes signature.
_vp, _i64, _int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
_FWD_ARGS = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _int, _vp, _vp, _i64, _i64, _i64, _i64,
             _int, _vp]
# sscan_fwd_ex: sscan_fwd's arguments with h0 and disc inserted after softplus_flag.
_FWD_EX_ARGS = _FWD_ARGS[:9] + [_vp, _int] + _FWD_ARGS[9:]
# sscan_step: u, delta, A, B, C, D, z, delta_bias, softplus, disc, h, y, batch, dim, N, dtype,
# stream.
_STEP_ARGS = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _int, _int, _vp, _vp, _i64, _i64, _i64,
              _int, _vp]
# sscan_conv1d_silu: x, w, bias, x_prev, silu, y, batch, L, dim, width, dtype, stream.
_CONV_ARGS = [_vp, _vp, _vp, _vp, _int, _vp, _i64, _i64, _i64, _i64, _int, _vp]
# sscan_bwd: the sscan_fwd_ex inputs (u .. disc), dy, dh_last, du, ddelta, dA, dB, dC, dD, dz,
# ddelta_bias, dh0, batch, L, dim, N, dtype, stream.
_BWD_ARGS = [_vp] * 9 + [_vp, _int] + [_vp] * 11 + [_i64] * 4 + [_int, _vp]
_BWD_ARGS[8] = _int  # softplus_flag


class Tuning(ctypes.Structure):
    """sscan_tuning_t (include/sscan_tuning.h): layout overrides and the fault-injection hook."""
    _fields_ = [("states_per_lane", ctypes.c_int), ("segments", ctypes.c_int),
                ("threads", ctypes.c_int), ("stages", ctypes.c_int), ("chunk", ctypes.c_int),
                ("force_plain", ctypes.c_int), ("bwd_segments", ctypes.c_int),
                ("conv_plain", ctypes.c_int), ("ctas_per_sm", ctypes.c_int),
                ("test_skip_publish", ctypes.c_int), ("time_scan", ctypes.c_int)]


_TUNING_P = ctypes.POINTER(Tuning)
SIGNATURES = {
    "sscan_fwd": (_FWD_ARGS, _int),
    "sscan_bwd": (_BWD_ARGS, _int),
    "sscan_conv1d_silu": (_CONV_ARGS, _int),
    "sscan_fwd_ex": (_FWD_EX_ARGS, _int),
    "sscan_step": (_STEP_ARGS, _int),
    "sscan_fwd_host": (_FWD_ARGS, _int),
    "sscan_fwd_noalloc": (_FWD_ARGS, _int),
    "sscan_get_device_error": ([_vp], _int),
    "sscan_status_string": ([_int], ctypes.c_char_p),
    "sscan_release": ([], _int),
    "sscan_set_tuning": ([_TUNING_P], _int),
    "sscan_get_tuning": ([_TUNING_P], _int),
    "sscan_exp2_accurate": ([_vp, _vp, _i64, _vp], _int),
}

_lib = None


class SscanError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS.get(code, code)}")
        self.code = code


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libsscan.so (raises OSError if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise OSError(f"libsscan.so not built at {p}; run selective_state_space_158_b300.build")
    lib = ctypes.CDLL(p)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    if path is None:
        _lib = lib
    return lib


def _check(code: int, where: str):
    if code != 0:
        raise SscanError(code, where)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SSCAN_F32
    if t.dtype == torch.bfloat16:
        return SSCAN_BF16
    raise TypeError(f"io tensors must be float32 or bfloat16, got {t.dtype}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def fwd(u: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
        C: torch.Tensor, D: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
        delta_bias: Optional[torch.Tensor] = None, softplus: bool = True,
        y: Optional[torch.Tensor] = None, h_last: Optional[torch.Tensor] = None,
        return_last_state: bool = True, stream=None, h0: Optional[torch.Tensor] = None,
        euler: bool = False):
    """Selective-scan forward on CUDA tensors (asynchronous on ``stream`` or the current stream).

    u, delta, z: (batch, L, dim); B, C: (batch, L, N) with 1 <= N <= 16, all of one io dtype
    (float32 or bfloat16); A: (dim, N) float32; D, delta_bias: (dim,) float32; h0: optional
    initial state (batch, dim, N) float32; ``euler`` selects the decay factor 1 + dt A.
    Calls ``sscan_fwd``, or ``sscan_fwd_ex`` when h0 or euler is given.
    Returns ``y`` (batch, L, dim) in the io dtype and, if ``return_last_state``, ``h_last``
    (batch, dim, N) float32.
    """
    lib = load()
    io = _dtype_code(u)
    batch, L, dim = u.shape
    N = B.shape[-1]
    dev = u.device
    if dev.type != "cuda":
        raise ValueError("libsscan computes on CUDA tensors only")
    for name, t, shape, dt in [("delta", delta, (batch, L, dim), u.dtype),
                               ("B", B, (batch, L, N), u.dtype), ("C", C, (batch, L, N), u.dtype),
                               ("A", A, (dim, N), torch.float32)]:
        if tuple(t.shape) != shape or t.dtype != dt or t.device != dev:
            raise ValueError(f"{name}: expected {shape} {dt} on {dev}, got "
                             f"{tuple(t.shape)} {t.dtype} on {t.device}")
    for name, t, shape, dt in [("D", D, (dim,), torch.float32), ("z", z, (batch, L, dim), u.dtype),
                               ("delta_bias", delta_bias, (dim,), torch.float32),
                               ("h0", h0, (batch, dim, N), torch.float32)]:
        if t is not None and (tuple(t.shape) != shape or t.dtype != dt or t.device != dev):
            raise ValueError(f"{name}: expected {shape} {dt} on {dev}")
    ts = [u, delta, A, B, C, D, z, delta_bias, h0]
    if any(t is not None and not t.is_contiguous() for t in ts):
        raise ValueError("all tensors must be contiguous")
    if y is None:
        y = torch.empty_like(u)
    if return_last_state and h_last is None:
        h_last = torch.empty((batch, dim, N), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        if h0 is None and not euler:
            where = "sscan_fwd"
            code = lib.sscan_fwd(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                 _ptr(z), _ptr(delta_bias), int(bool(softplus)), _ptr(y),
                                 _ptr(h_last), batch, L, dim, N, io, _stream_handle(stream, dev))
        else:
            where = "sscan_fwd_ex"
            code = lib.sscan_fwd_ex(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                    _ptr(z), _ptr(delta_bias), int(bool(softplus)), _ptr(h0),
                                    SSCAN_DISC_EULER if euler else SSCAN_DISC_ZOH, _ptr(y),
                                    _ptr(h_last), batch, L, dim, N, io,
                                    _stream_handle(stream, dev))
    _check(code, where)
    return (y, h_last) if return_last_state else y


def step(u: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
         C: torch.Tensor, h: torch.Tensor, D: Optional[torch.Tensor] = None,
         z: Optional[torch.Tensor] = None, delta_bias: Optional[torch.Tensor] = None,
         softplus: bool = True, euler: bool = False, y: Optional[torch.Tensor] = None,
         stream=None) -> torch.Tensor:
    """One recurrence step for every (batch, channel) through ``sscan_step``.

    u, delta, z: (batch, dim); B, C: (batch, N), one io dtype; A: (dim, N) float32; h: (batch,
    dim, N) float32 state, updated in place. Returns y (batch, dim) in the io dtype.
    """
    lib = load()
    io = _dtype_code(u)
    batch, dim = u.shape
    N = B.shape[-1]
    dev = u.device
    if dev.type != "cuda":
        raise ValueError("libsscan computes on CUDA tensors only")
    for name, t, shape, dt in [("delta", delta, (batch, dim), u.dtype),
                               ("B", B, (batch, N), u.dtype), ("C", C, (batch, N), u.dtype),
                               ("A", A, (dim, N), torch.float32),
                               ("h", h, (batch, dim, N), torch.float32)]:
        if tuple(t.shape) != shape or t.dtype != dt or t.device != dev:
            raise ValueError(f"{name}: expected {shape} {dt} on {dev}")
    for name, t, shape, dt in [("D", D, (dim,), torch.float32), ("z", z, (batch, dim), u.dtype),
                               ("delta_bias", delta_bias, (dim,), torch.float32)]:
        if t is not None and (tuple(t.shape) != shape or t.dtype != dt or t.device != dev):
            raise ValueError(f"{name}: expected {shape} {dt} on {dev}")
    if any(t is not None and not t.is_contiguous() for t in [u, delta, A, B, C, h, D, z,
                                                              delta_bias]):
        raise ValueError("all tensors must be contiguous")
    if y is None:
        y = torch.empty_like(u)
    with torch.cuda.device(dev):
        code = lib.sscan_step(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                              _ptr(delta_bias), int(bool(softplus)),
                              SSCAN_DISC_EULER if euler else SSCAN_DISC_ZOH, _ptr(h), _ptr(y),
                              batch, dim, N, io, _stream_handle(stream, dev))
    _check(code, "sscan_step")
    return y


def fwd_host(u: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
             C: torch.Tensor, D=None, z=None, delta_bias=None, softplus: bool = True,
             y: Optional[torch.Tensor] = None, h_last: Optional[torch.Tensor] = None,
             device: int = 0, stream=None):
    """The same operation on CPU tensors (pinned memory recommended): the library copies the
    inputs to ``device``, scans, copies y and h_last back and synchronizes. Returns (y, h_last)."""
    lib = load()
    io = _dtype_code(u)
    batch, L, dim = u.shape
    N = B.shape[-1]
    ts = [u, delta, A, B, C, D, z, delta_bias]
    if any(t is not None and (t.device.type != "cpu" or not t.is_contiguous()) for t in ts):
        raise ValueError("fwd_host takes contiguous CPU tensors")
    if y is None:
        y = torch.empty_like(u)
    if h_last is None:
        h_last = torch.empty((batch, dim, N), dtype=torch.float32)
    dev = torch.device("cuda", device)
    with torch.cuda.device(dev):
        code = lib.sscan_fwd_host(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                  _ptr(z), _ptr(delta_bias), int(bool(softplus)), _ptr(y),
                                  _ptr(h_last), batch, L, dim, N, io,
                                  _stream_handle(stream, dev))
    _check(code, "sscan_fwd_host")
    return y, h_last


def bwd(u: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
        C: torch.Tensor, dy: torch.Tensor, D: Optional[torch.Tensor] = None,
        z: Optional[torch.Tensor] = None, delta_bias: Optional[torch.Tensor] = None,
        dh_last: Optional[torch.Tensor] = None, softplus: bool = True,
        h0: Optional[torch.Tensor] = None, euler: bool = False, want_dh0: bool = False,
        stream=None) -> dict:
    """Gradients of sum(dy * y) + sum(dh_last * h_last) through ``sscan_bwd``.

    Forward inputs as for ``fwd``; dy like u; dh_last (batch, dim, N) float32 or None.
    Returns a dict: du, ddelta (io dtype), dA, dB, dC (float32), and dD / dz / ddelta_bias when
    D / z / delta_bias are given, dh0 when ``want_dh0``.
    """
    lib = load()
    io = _dtype_code(u)
    batch, L, dim = u.shape
    N = B.shape[-1]
    dev = u.device
    if dev.type != "cuda":
        raise ValueError("libsscan computes on CUDA tensors only")
    if tuple(dy.shape) != (batch, L, dim) or dy.dtype != u.dtype:
        raise ValueError("dy must match u")
    ts = [u, delta, A, B, C, D, z, delta_bias, h0, dy, dh_last]
    if any(t is not None and (not t.is_contiguous() or t.device != dev) for t in ts):
        raise ValueError("all tensors must be contiguous and on u's device")
    f32 = dict(dtype=torch.float32, device=dev)
    g = {"du": torch.empty_like(u), "ddelta": torch.empty_like(u),
         "dA": torch.empty((dim, N), **f32), "dB": torch.empty((batch, L, N), **f32),
         "dC": torch.empty((batch, L, N), **f32)}
    if D is not None:
        g["dD"] = torch.empty((dim,), **f32)
    if z is not None:
        g["dz"] = torch.empty_like(u)
    if delta_bias is not None:
        g["ddelta_bias"] = torch.empty((dim,), **f32)
    if want_dh0:
        g["dh0"] = torch.empty((batch, dim, N), **f32)
    with torch.cuda.device(dev):
        code = lib.sscan_bwd(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                             _ptr(delta_bias), int(bool(softplus)), _ptr(h0),
                             SSCAN_DISC_EULER if euler else SSCAN_DISC_ZOH, _ptr(dy),
                             _ptr(dh_last), _ptr(g["du"]), _ptr(g["ddelta"]), _ptr(g["dA"]),
                             _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g.get("dD")), _ptr(g.get("dz")),
                             _ptr(g.get("ddelta_bias")), _ptr(g.get("dh0")), batch, L, dim, N,
                             io, _stream_handle(stream, dev))
    _check(code, "sscan_bwd")
    return g


def conv1d_silu(x: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor] = None,
                x_prev: Optional[torch.Tensor] = None, silu: bool = True,
                y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Causal depthwise convolution over time + SiLU through ``sscan_conv1d_silu``.

    x: (batch, L, dim) float32 or bfloat16; w: (dim, width) float32; bias: (dim,) float32;
    x_prev: (batch, width - 1, dim) in x's dtype (inputs before t = 0). Returns y like x.
    """
    lib = load()
    io = _dtype_code(x)
    batch, L, dim = x.shape
    width = w.shape[-1]
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("libsscan computes on CUDA tensors only")
    if tuple(w.shape) != (dim, width) or w.dtype != torch.float32 or w.device != dev:
        raise ValueError(f"w: expected ({dim}, width) float32 on {dev}")
    if bias is not None and (tuple(bias.shape) != (dim,) or bias.dtype != torch.float32):
        raise ValueError("bias: expected (dim,) float32")
    if x_prev is not None and (tuple(x_prev.shape) != (batch, width - 1, dim) or
                               x_prev.dtype != x.dtype):
        raise ValueError(f"x_prev: expected {(batch, width - 1, dim)} {x.dtype}")
    if any(t is not None and not t.is_contiguous() for t in [x, w, bias, x_prev]):
        raise ValueError("all tensors must be contiguous")
    if y is None:
        y = torch.empty_like(x)
    with torch.cuda.device(dev):
        code = lib.sscan_conv1d_silu(_ptr(x), _ptr(w), _ptr(bias), _ptr(x_prev),
                                     int(bool(silu)), _ptr(y), batch, L, dim, width, io,
                                     _stream_handle(stream, dev))
    _check(code, "sscan_conv1d_silu")
    return y


def device_error(stream=None, device=None) -> int:
    """Synchronize and return (then clear) the device status word; 0 means no device error."""
    lib = load()
    dev = device if device is not None else torch.cuda.current_device()
    with torch.cuda.device(dev):
        return lib.sscan_get_device_error(_stream_handle(stream, dev))


@contextlib.contextmanager
def tuning(**fields):
    """Within the block, the library uses the given layout overrides (fields of
    ``sscan_tuning_t``; the others keep their automatic choice); the previous setting is restored
    on exit. For tests and tuning sweeps."""
    lib = load()
    prev = Tuning()
    _check(lib.sscan_get_tuning(ctypes.byref(prev)), "sscan_get_tuning")
    t = Tuning(test_skip_publish=-1)
    for k, v in fields.items():
        if k not in dict(Tuning._fields_):
            raise KeyError(f"unknown tuning field {k}")
        setattr(t, k, int(v))
    _check(lib.sscan_set_tuning(ctypes.byref(t)), "sscan_set_tuning")
    try:
        yield
    finally:
        _check(lib.sscan_set_tuning(ctypes.byref(prev)), "sscan_set_tuning")


def exp2_accurate(x: torch.Tensor, stream=None) -> torch.Tensor:
    """2^x with the library's accurate exponential (``sscan_exp2_accurate``); float32 CUDA."""
    lib = load()
    if x.dtype != torch.float32 or x.device.type != "cuda" or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 CUDA tensor")
    y = torch.empty_like(x)
    with torch.cuda.device(x.device):
        code = lib.sscan_exp2_accurate(_ptr(x), _ptr(y), x.numel(),
                                       _stream_handle(stream, x.device))
    _check(code, "sscan_exp2_accurate")
    return y


def status_string(code: int) -> str:
    return load().sscan_status_string(code).decode()
