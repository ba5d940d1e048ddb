"""The C ABI library loads without a GPU and exports every symbol include/sscan.h declares;
argument errors come back synchronously, before any CUDA call."""
import ctypes
import os
import re

import pytest

from selective_state_space_158_b300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*[\w\s\*]+?\b(sscan_\w+)\s*\(", text, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = declared_functions()
    assert {"sscan_fwd", "sscan_fwd_host", "sscan_get_device_error", "sscan_status_string",
            "sscan_release"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
        assert n in binding.SIGNATURES, f"{n} has no binding signature"


def test_status_strings(lib):
    assert binding.status_string(0) == "SSCAN_OK"
    assert binding.status_string(4) == "SSCAN_ERR_CARRY_TIMEOUT"
    assert binding.status_string(99) == "SSCAN_ERR_UNKNOWN"


def test_argument_errors_are_synchronous_without_a_device(lib):
    dummy = ctypes.c_void_p(256)  # never dereferenced: the checks fail first
    ok = [dummy, dummy, dummy, dummy, dummy, None, None, None, 1, dummy, None, 1, 8, 64, 16, 0,
          None]
    for idx, val in [(14, 0), (14, 17), (12, -1), (11, -2), (13, -1), (15, 3), (0, None),
                     (2, None), (9, None), (3, None)]:
        args = list(ok)
        args[idx] = val
        assert lib.sscan_fwd(*args) == 1, (idx, val)
        assert lib.sscan_fwd_host(*args) == 1, (idx, val)
    # size products that overflow int64
    args = list(ok)
    args[11], args[12], args[13] = 1 << 40, 1 << 40, 64
    assert lib.sscan_fwd(*args) == 1
    # sscan_fwd_ex: the same checks, plus an out-of-range decay-factor selector
    ok_ex = ok[:9] + [None, 0] + ok[9:]
    for idx, val in [(16, 0), (16, 17), (14, -1), (2, None), (11, None), (10, 2), (10, -1)]:
        args = list(ok_ex)
        args[idx] = val
        assert lib.sscan_fwd_ex(*args) == 1, (idx, val)
    # sscan_step: u, delta, A, B, C, D, z, bias, softplus, disc, h, y, batch, dim, N, dtype, stream
    ok_st = [dummy, dummy, dummy, dummy, dummy, None, None, None, 1, 0, dummy, dummy, 4, 64, 16,
             0, None]
    for idx, val in [(14, 0), (14, 17), (12, -1), (13, -1), (15, 2), (9, 5), (10, None),
                     (11, None), (0, None), (2, None)]:
        args = list(ok_st)
        args[idx] = val
        assert lib.sscan_step(*args) == 1, (idx, val)
    # sscan_conv1d_silu: x, w, bias, x_prev, silu, y, batch, L, dim, width, dtype, stream
    other = ctypes.c_void_p(512)
    ok_cv = [dummy, dummy, None, None, 1, other, 2, 16, 64, 4, 0, None]
    for idx, val in [(9, 0), (9, 65), (6, -1), (7, -1), (8, -1), (10, 2), (0, None), (1, None),
                     (5, None), (5, dummy)]:  # the last: y aliasing x
        args = list(ok_cv)
        args[idx] = val
        assert lib.sscan_conv1d_silu(*args) == 1, (idx, val)


def test_tuning_ranges_are_checked_without_a_device(lib):
    """sscan_set_tuning refuses out-of-range fields and leaves the setting unchanged; the
    setting round-trips through sscan_get_tuning; NULL restores every automatic choice."""
    T = binding.Tuning
    bad = [dict(states_per_lane=3), dict(threads=48), dict(threads=288), dict(stages=1),
           dict(stages=9), dict(chunk=8), dict(ctas_per_sm=33), dict(test_skip_publish=-2),
           dict(time_scan=3), dict(time_scan=-1), dict(segments=-1)]
    for fields in bad:
        t = T(test_skip_publish=-1)
        for k, v in fields.items():
            setattr(t, k, v)
        assert lib.sscan_set_tuning(ctypes.byref(t)) == 1, fields
    good = T(states_per_lane=8, segments=3, threads=96, stages=4, chunk=16, ctas_per_sm=2,
             test_skip_publish=-1, time_scan=2)
    assert lib.sscan_set_tuning(ctypes.byref(good)) == 0
    back = T()
    assert lib.sscan_get_tuning(ctypes.byref(back)) == 0
    for name, _ in T._fields_:
        assert getattr(back, name) == getattr(good, name), name
    assert lib.sscan_set_tuning(None) == 0
    assert lib.sscan_get_tuning(ctypes.byref(back)) == 0
    assert (back.states_per_lane, back.segments, back.time_scan, back.test_skip_publish) == \
        (0, 0, 0, -1)
