"""The allocation-free entry point, sscan_fwd_noalloc.

Some callers cannot allocate device memory when they run the scan: a framework or caching
allocator owns all of it, or their path may not risk the synchronisation or the failure that an
allocation can bring. For them sscan_fwd_noalloc keeps its scratch (fp32 copies of B and C, the
chunk-carry flags and segment summaries) in a fixed static device array instead of a
stream-ordered allocation.

These tests call it through the C ABI, twice in a row, on shapes that use the scratch (a
sequence split across thread blocks, and bf16 B/C that are widened), and check each result
against the fp64 oracle under the parity tolerance and against sscan_fwd's result on the same
inputs (the same kernels: bitwise equal). They check that the calls leave the device's memory
untouched (free memory and the default pool's use), that a call needing more scratch than the
array holds is refused before anything is launched, and that the entry point honours the same
kernel-path choice as sscan_fwd.

This file is collected last on purpose: if it fails, a run that stops at the first failure has
already run every other test. It also passes when run alone in a fresh process.
"""
import ctypes

import pytest
import torch

from parity import assert_within, compare, oracle_full
from selective_state_space_158_b300 import binding
from selective_state_space_158_b300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


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


def _pool_used_bytes():
    """Bytes in use from the device's default stream-ordered pool (None if the query is not
    available in this environment)."""
    try:
        from cuda.bindings import runtime as rt
    except ImportError:
        return None
    err, pool = rt.cudaDeviceGetDefaultMemPool(0)
    if err != rt.cudaError_t.cudaSuccess:
        return None
    err, used = rt.cudaMemPoolGetAttribute(pool, rt.cudaMemPoolAttr.cudaMemPoolAttrUsedMemCurrent)
    return int(used) if err == rt.cudaError_t.cudaSuccess else None


@pytest.mark.parametrize("key", ["fp32", "long"])
def test_noalloc_matches_oracle_and_sscan_fwd_twice_in_a_row(key, tune):
    tune(segments=6)  # split the sequence: the chunk-carry part of the static scratch is used
    w = WORKLOADS[key].replace(batch=2, L=4096, dim=128)
    x = make_inputs(w, device=DEV)
    y_ref, h_ref = binding.fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x.get("D"),
                               x.get("z"), x.get("delta_bias"))
    assert binding.device_error() == 0
    yr, hr, ym = oracle_full(x)
    lib = binding.load()
    y = torch.empty_like(x["u"])
    h = torch.empty_like(h_ref)
    assert _noalloc(lib, x, y, h) == 0  # warm-up: the first call on a device does its set-up
    for call in range(2):
        y.fill_(float("nan"))
        h.fill_(float("nan"))
        # Free device memory and the default pool's use are read right around the call: the
        # checks in between (torch's own temporaries) may grow torch's cache.
        torch.cuda.synchronize()
        free0, used0 = torch.cuda.mem_get_info()[0], _pool_used_bytes()
        assert _noalloc(lib, x, y, h) == 0, f"call {call}"
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0, f"call {call} changed free device memory"
        assert _pool_used_bytes() == used0, f"call {call} used the default pool"
        assert binding.device_error() == 0
        assert_within(compare(y, h, yr, hr, w.io, y_mag=ym), w.io, f"noalloc call {call} vs oracle")
        assert torch.equal(y, y_ref) and torch.equal(h, h_ref), f"call {call} vs sscan_fwd"


def test_noalloc_plain_load_path(tune):
    """With the plain-load kernel forced (as sscan_fwd honours it), the entry point runs it."""
    tune(force_plain=1)
    w = WORKLOADS["bf16"].replace(batch=2, L=77, dim=40)
    x = make_inputs(w, device=DEV)
    y = torch.empty_like(x["u"])
    h = torch.empty((2, 40, 16), dtype=torch.float32, device=DEV)
    assert _noalloc(binding.load(), x, y, h) == 0
    assert binding.device_error() == 0
    yr, hr, ym = oracle_full(x)
    assert_within(compare(y, h, yr, hr, w.io, y_mag=ym), w.io, "noalloc plain-load path")
    y2, h2 = binding.fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                         x["delta_bias"])
    assert torch.equal(y, y2) and torch.equal(h, h2)


def test_noalloc_refuses_a_call_that_needs_more_scratch(tune):
    tune(segments=64)  # 64 segments x 4096 channels: far above the array's 16 MiB
    w = WORKLOADS["long"].replace(batch=1, L=4096, dim=4096)
    x = make_inputs(w, device=DEV)
    y = torch.empty_like(x["u"])
    h = torch.empty((1, 4096, 16), dtype=torch.float32, device=DEV)
    assert _noalloc(binding.load(), x, y, h) == 5  # SSCAN_ERR_SCRATCH_TOO_SMALL
    assert binding.status_string(5) == "SSCAN_ERR_SCRATCH_TOO_SMALL"
