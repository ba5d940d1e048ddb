"""GPU parity: libsscan (through its C ABI) against the fp64 oracle on the same seeded inputs.

Small shapes are compared element by element over whole tensors; they span several channel
tiles and time chunks with ragged tails, every kernel layout, the chunk carry and the optional
operands. The full-size workloads are in test_gpu_fullsize.py.
"""
import pytest
import torch

from parity import assert_within, compare, oracle_full
from selective_state_space_158_b300 import binding
from selective_state_space_158_b300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
STATES_PER_LANE = [16, 8, 4]  # one, two or four lanes per channel


def run_lib(x, softplus=True):
    y, h = binding.fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x.get("D"), x.get("z"),
                       x.get("delta_bias"), softplus=softplus)
    assert binding.device_error() == 0
    return y, h


def check_full(w, x=None, softplus=True, what=""):
    x = x if x is not None else make_inputs(w, device=DEV)
    y, h = run_lib(x, softplus)
    yr, hr, ym = oracle_full(x, softplus)
    res = compare(y, h, yr, hr, w.io, y_mag=ym)
    assert_within(res, w.io, what or w.name)
    return res


# ---- small whole-tensor cases -----------------------------------------------------------------

def test_tiny_workload_whole_tensor():
    check_full(WORKLOADS["tiny"])


@pytest.mark.parametrize("K", STATES_PER_LANE)
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_ragged_shapes_each_lane_shape(K, io, tune):
    """L not a multiple of the chunk, dim not a multiple of the channel tile, z/D/bias on."""
    tune(states_per_lane=K)
    base = WORKLOADS["fp32"] if io == "f32" else WORKLOADS["bf16"]
    w = base.replace(batch=2, L=301, dim=200 if io == "f32" else 136)
    check_full(w, what=f"K={K} {io}")


@pytest.mark.parametrize("segments", [2, 3, 5, 19])
@pytest.mark.parametrize("K", STATES_PER_LANE)
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_chunk_carry_segments(segments, K, io, tune):
    """The sequence split into time segments run by different CTAs (decoupled look-back)."""
    tune(states_per_lane=K, segments=segments)
    base = WORKLOADS["fp32"] if io == "f32" else WORKLOADS["long"]
    w = base.replace(batch=2, L=301, dim=136)
    check_full(w, what=f"segments={segments} K={K} {io}")


def test_chunk_carry_long_sequence_small_width(tune):
    """Many segments over a long sequence with few channels (the long workload's regime), in
    the lane kernel (the time-lane kernel would be chosen for this shape)."""
    tune(time_scan=2)
    w = WORKLOADS["long"].replace(L=1 << 14, dim=64)
    check_full(w, what="long L, narrow")


def test_chunk_carry_timeout_reports_status_and_context_survives(tune):
    """A segment that never publishes makes its successors' bounded look-back waits run out:
    the call finishes, the device status word says SSCAN_ERR_CARRY_TIMEOUT, and the next call
    on the same context is correct again."""
    tune(segments=3, test_skip_publish=0, time_scan=2)  # the lane kernel's carry
    w = WORKLOADS["fp32"].replace(batch=1, L=200, dim=64)
    x = make_inputs(w, device=DEV)
    binding.fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"])
    assert binding.device_error() == 4
    assert binding.device_error() == 0  # reading clears it
    tune(segments=3, time_scan=2)
    check_full(w, x=x, what="after timeout")


@pytest.mark.parametrize("stages,threads", [(2, 64), (3, 128), (4, 128), (2, 256), (3, 32)])
def test_pipeline_and_cta_shape_invariance(stages, threads, tune):
    tune(stages=stages, threads=threads)
    w = WORKLOADS["fp32"].replace(batch=2, L=257, dim=256)
    check_full(w, what=f"stages={stages} threads={threads}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_plain_load_path(io, tune):
    tune(force_plain=1)
    base = WORKLOADS["fp32"] if io == "f32" else WORKLOADS["bf16"]
    check_full(base.replace(batch=2, L=77, dim=40), what=f"simple {io}")


@pytest.mark.parametrize("dim,N", [(37, 16), (40, 5), (64, 8), (64, 4), (33, 1)])
def test_unaligned_and_small_state(dim, N):
    w = WORKLOADS["fp32"].replace(batch=2, L=65, dim=dim, N=N)
    check_full(w, what=f"dim={dim} N={N}")


@pytest.mark.parametrize("flags", [dict(has_z=False), dict(has_D=False), dict(has_bias=False),
                                   dict(has_z=False, has_D=False, has_bias=False)])
def test_optional_operands(flags):
    w = WORKLOADS["bf16"].replace(batch=2, L=100, dim=64, **flags)
    check_full(w, what=str(flags))


def test_softplus_off():
    w = WORKLOADS["fp32"].replace(batch=1, L=90, dim=64)
    x = make_inputs(w, device=DEV)
    x["delta"] = torch.nn.functional.softplus(x["delta"].double() + x["delta_bias"].double()).float()
    x["delta_bias"] = None
    check_full(w, x=x, softplus=False, what="softplus off")


@pytest.mark.parametrize("L", [1, 2, 31, 32, 33])
def test_short_sequences(L):
    check_full(WORKLOADS["fp32"].replace(batch=3, L=L, dim=64), what=f"L={L}")


def test_empty_inputs():
    w = WORKLOADS["fp32"].replace(batch=2, L=0, dim=64)
    x = make_inputs(w, device=DEV)
    h = torch.full((2, 64, 16), 7.0, device=DEV)
    y, h = binding.fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                       x["delta_bias"], h_last=h)
    torch.cuda.synchronize()
    assert y.numel() == 0 and torch.all(h == 0)
    w0 = WORKLOADS["fp32"].replace(batch=0, L=16, dim=64)
    x0 = make_inputs(w0, device=DEV)
    y0, _ = binding.fwd(x0["u"], x0["delta"], x0["A"], x0["B"], x0["C"])
    assert y0.numel() == 0


# ---- hygiene: every output written, nothing else touched, deterministic -----------------------

def test_outputs_fully_written_and_guard_band_untouched():
    w = WORKLOADS["bf16"].replace(batch=2, L=130, dim=72)
    x = make_inputs(w, device=DEV)
    n = 2 * 130 * 72
    guard = 4096
    buf = torch.full((n + 2 * guard,), float("nan"), dtype=torch.bfloat16, device=DEV)
    buf[:guard] = 3.0
    buf[-guard:] = 3.0
    y = buf[guard:guard + n].view(2, 130, 72)
    hb = torch.full((2 * 72 * 16 + 2 * guard,), 5.0, device=DEV)
    h = hb[guard:-guard].view(2, 72, 16)
    h.fill_(float("nan"))
    binding.fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
                y=y, h_last=h)
    torch.cuda.synchronize()
    assert not torch.isnan(y).any() and not torch.isnan(h).any()
    assert torch.all(buf[:guard] == 3.0) and torch.all(buf[-guard:] == 3.0)
    assert torch.all(hb[:guard] == 5.0) and torch.all(hb[-guard:] == 5.0)


def test_bitwise_deterministic():
    w = WORKLOADS["fp32"].replace(batch=2, L=500, dim=256)
    x = make_inputs(w, device=DEV)
    y1, h1 = run_lib(x)
    y2, h2 = run_lib(x)
    assert torch.equal(y1, y2) and torch.equal(h1, h2)


def _rows(x, r0, r1):
    return {k: (v[r0:r1].contiguous() if v is not None and v.dim() == 3 and k != "A" else v)
            for k, v in x.items()}


def test_host_entry_matches_device_entry():
    """The host entry cuts a batch of up to 8 rows into one-row slices: each equals the device
    entry run on that row alone."""
    w = WORKLOADS["fp32"].replace(batch=2, L=200, dim=128)
    x = make_inputs(w, device=DEV)
    xc = {k: (v.cpu().pin_memory() if v is not None else None) for k, v in x.items()}
    yh, hh = binding.fwd_host(xc["u"], xc["delta"], xc["A"], xc["B"], xc["C"], xc["D"], xc["z"],
                              xc["delta_bias"])
    for r in range(w.batch):
        y, h = run_lib(_rows(x, r, r + 1))
        assert torch.equal(yh[r:r + 1], y.cpu()) and torch.equal(hh[r:r + 1], h.cpu()), r


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_host_entry_many_slices(io):
    """19 batch rows: slices of 3 rows rotating over the library's streams, against the
    oracle."""
    base = WORKLOADS["fp32"] if io == "f32" else WORKLOADS["bf16"]
    w = base.replace(batch=19, L=150, dim=64)
    x = make_inputs(w, device=DEV)
    xc = {k: (v.cpu().pin_memory() if v is not None else None) for k, v in x.items()}
    yh, hh = binding.fwd_host(xc["u"], xc["delta"], xc["A"], xc["B"], xc["C"], xc["D"], xc["z"],
                              xc["delta_bias"])
    yr, hr, ym = oracle_full(x)
    assert_within(compare(yh, hh, yr, hr, w.io, y_mag=ym), w.io, f"host entry, 19 rows, {io}")


@pytest.mark.parametrize("io,batch", [("f32", 1), ("bf16", 3)])
def test_host_entry_time_slices(io, batch):
    """Few batch rows and a long sequence: the host entry cuts the sequence into time slices
    (each continuing from the previous one's end state, staged as dense (batch, slice, dim)
    blocks by strided copies), against the oracle over the whole sequence."""
    base = WORKLOADS["fp32"] if io == "f32" else WORKLOADS["bf16"]
    w = base.replace(batch=batch, L=50001, dim=24)
    x = make_inputs(w, device=DEV)
    xc = {k: (v.cpu().pin_memory() if v is not None else None) for k, v in x.items()}
    yh, hh = binding.fwd_host(xc["u"], xc["delta"], xc["A"], xc["B"], xc["C"], xc["D"], xc["z"],
                              xc["delta_bias"])
    yr, hr, ym = oracle_full(x)
    assert_within(compare(yh, hh, yr, hr, w.io, y_mag=ym), w.io, f"host entry, time slices, {io}")


def test_invalid_arguments_rejected_synchronously():
    w = WORKLOADS["fp32"].replace(batch=1, L=8, dim=64)
    x = make_inputs(w, device=DEV)
    lib = binding.load()
    p = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    y = torch.empty_like(x["u"])
    args = [p(x["u"]), p(x["delta"]), p(x["A"]), p(x["B"]), p(x["C"]), None, None, None, 1,
            p(y), None, 1, 8, 64, 16, 0, None]
    bad = list(args)
    bad[14] = 17  # N > 16
    assert lib.sscan_fwd(*bad) == 1
    bad = list(args)
    bad[0] = None  # u missing
    assert lib.sscan_fwd(*bad) == 1
    bad = list(args)
    bad[15] = 7  # unknown dtype
    assert lib.sscan_fwd(*bad) == 1
    bad = list(args)
    bad[12] = -1  # negative L
    assert lib.sscan_fwd(*bad) == 1
    assert lib.sscan_fwd(*args) == 0
    torch.cuda.synchronize()
