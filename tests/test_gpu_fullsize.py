"""Full-size parity: the workloads at their full shapes, in the launch configuration the
benchmark times, against the fp64 oracle over whole tensors: every output element of y and
h_last, every channel and every step.

The long sequence (batch 1, L 2^20, D 1536, the chunk carry across many time segments) is
compared in blocks of 256 channels, so that the host holds one block's fp64 oracle output at a
time; the error metric's rms is taken over each block.
"""
import pytest
import torch

from parity import assert_within, compare, oracle_full
from selective_state_space_158_b300 import binding
from selective_state_space_158_b300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _run(x):
    y, h = binding.fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x.get("D"), x.get("z"),
                       x.get("delta_bias"))
    assert binding.device_error() == 0
    return y, h


@pytest.mark.parametrize("key", ["fp32", "bf16", "wide"])
def test_full_size_whole_tensor(key):
    w = WORKLOADS[key]
    x = make_inputs(w, device=DEV)
    y, h = _run(x)
    yr, hr, ym = oracle_full(x)
    res = compare(y, h, yr, hr, w.io, y_mag=ym)
    print(key, {k: {kk: f"{vv:.3g}" for kk, vv in v.items()} for k, v in res.items()})
    assert_within(res, w.io, w.name)
    del x, y, h
    torch.cuda.empty_cache()


def test_long_sequence_whole_tensor_in_channel_blocks():
    w = WORKLOADS["long"]
    x = make_inputs(w, device=DEV)
    y, h = _run(x)
    blk = 256
    for c0 in range(0, w.dim, blk):
        c1 = min(w.dim, c0 + blk)
        xs = {}
        for k, v in x.items():
            if v is None:
                xs[k] = None
            elif k in ("u", "delta", "z"):
                xs[k] = v[:, :, c0:c1].contiguous()
            elif k in ("A", "D", "delta_bias"):
                xs[k] = v[c0:c1].contiguous()
            else:  # B, C: shared over channels
                xs[k] = v
        yr, hr, ym = oracle_full(xs)
        res = compare(y[:, :, c0:c1], h[:, c0:c1], yr, hr, w.io, y_mag=ym)
        print(f"long channels {c0}..{c1 - 1}",
              {k: {kk: f"{vv:.3g}" for kk, vv in v.items()} for k, v in res.items()})
        assert_within(res, w.io, f"{w.name}, channels {c0}..{c1 - 1}")
        del xs, yr, hr
    del x, y, h
    torch.cuda.empty_cache()
