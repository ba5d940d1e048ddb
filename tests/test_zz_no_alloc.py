"""The allocation-free entry point, sscan_fwd_noalloc.

Some callers cannot allocate device memory when they run the scan (a framework or caching
allocator owns all of it, or an allocation's possible synchronisation is not allowed on their
path). For them sscan_fwd_noalloc keeps the chunk-carry scratch in a fixed static device array
instead of a stream-ordered allocation. These tests call it through the C ABI on a shape whose
sequence is split across thread blocks (so the scratch is really used), twice in a row, and
compare each result with sscan_fwd's under the parity tolerance; and they check that a call
needing more scratch than the array holds is refused before anything is launched.

This file is collected last on purpose: if it fails, a run that stops at the first failure has
already run every other test. It also passes when run alone in a fresh process.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

from parity import assert_within, err_stats, round_bf16
from selective_state_space_158_b300 import binding
from selective_state_space_158_b300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _segments_env():
    saved = os.environ.get("SSCAN_SEGMENTS")
    yield
    if saved is None:
        os.environ.pop("SSCAN_SEGMENTS", None)
    else:
        os.environ["SSCAN_SEGMENTS"] = saved


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, x, y, h):
    u = x["u"]
    batch, L, dim = u.shape
    N = x["B"].shape[-1]
    io = binding.SSCAN_F32 if u.dtype == torch.float32 else binding.SSCAN_BF16
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.sscan_fwd_noalloc(_p(u), _p(x["delta"]), _p(x["A"]), _p(x["B"]), _p(x["C"]),
                                 _p(x.get("D")), _p(x.get("z")), _p(x.get("delta_bias")), 1,
                                 _p(y), _p(h), batch, L, dim, N, io, stream)


@pytest.mark.parametrize("key", ["fp32", "long"])
def test_noalloc_matches_sscan_fwd_twice_in_a_row(key):
    os.environ["SSCAN_SEGMENTS"] = "6"  # split the sequence: the static scratch is used
    w = WORKLOADS[key].replace(batch=2, L=4096, dim=128)
    x = make_inputs(w, device=DEV)
    y_ref, h_ref = binding.fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x.get("D"),
                               x.get("z"), x.get("delta_bias"))
    assert binding.device_error() == 0
    lib = binding.load()
    yr = y_ref.double().cpu().numpy()
    hr = h_ref.double().cpu().numpy()
    for call in range(2):
        y = torch.full_like(x["u"], float("nan"))
        h = torch.full_like(h_ref, float("nan"))
        assert _noalloc(lib, x, y, h) == 0, f"call {call}"
        assert binding.device_error() == 0
        yg = y.double().cpu().numpy()
        ref = round_bf16(yr) if w.io == "bf16" else yr
        res = {"y": err_stats(yg, ref), "h": err_stats(h.double().cpu().numpy(), hr)}
        assert_within(res, w.io, f"noalloc call {call}")


def test_noalloc_refuses_a_call_that_needs_more_scratch():
    os.environ["SSCAN_SEGMENTS"] = "64"  # 64 segments x 4096 channels: far above 16 MiB
    w = WORKLOADS["long"].replace(batch=1, L=4096, dim=4096)
    x = make_inputs(w, device=DEV)
    y = torch.empty_like(x["u"])
    h = torch.empty((1, 4096, 16), dtype=torch.float32, device=DEV)
    assert _noalloc(binding.load(), x, y, h) == 5  # SSCAN_ERR_SCRATCH_TOO_SMALL
    assert binding.status_string(5) == "SSCAN_ERR_SCRATCH_TOO_SMALL"
