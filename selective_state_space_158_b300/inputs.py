"""Seeded synthetic inputs for the selective-scan forward.

This module is shared by the tests, the smoke check and the benchmark, on both sides of every
parity comparison: the CUDA library and the fp64 oracle read the very same tensors. It holds
none of the scan's arithmetic -- only random draws and the recipe that shapes them.

Recipe (every workload):
  * u, B, C, z and delta_raw are i.i.d. N(0, 1);
  * Dskip[d] ~ N(0, 1);
  * A[d, n] = -(n + 1) (the S4D-real pattern), or A[d, n] = -exp(U(log 1, log 16)) per (d, n);
  * a workload's "step range" [lo, hi] fixes the bias: per channel a base step
    dt0[d] = exp(U(log lo, log hi)) is drawn and delta_bias[d] is the value whose softplus is
    dt0[d], i.e. dt0 + log(-expm1(-dt0)). The effective step softplus(delta_raw + bias) then
    spreads around dt0.
  * bf16 workloads round each fp32 draw to bf16 (round to nearest even); A, Dskip and
    delta_bias stay fp32.

Each tensor draws from its own torch.Generator whose seed is derived from the workload seed and
the tensor's name, so a tensor does not depend on which others are drawn. Large workloads are
drawn directly on the GPU (the oracle then reads back only the channels it checks).
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    key: str
    name: str
    batch: int
    L: int
    dim: int
    N: int
    io: str  # "f32" or "bf16"
    A_kind: str  # "neg_n1" (A = -(n+1)) or "neg_exp_u" (A = -exp(U(log 1, log 16)))
    dt_range: tuple
    has_z: bool
    has_D: bool
    has_bias: bool = True
    softplus: bool = True
    seed_index: int = 0

    @property
    def elems(self) -> int:
        """B*L*D*N: the number of (batch, step, channel, state) updates."""
        return self.batch * self.L * self.dim * self.N

    def io_bytes(self) -> int:
        """Algorithmic HBM bytes of one forward: every input read once, every output written once."""
        s = 4 if self.io == "f32" else 2
        bld = self.batch * self.L * self.dim
        bln = self.batch * self.L * self.N
        nread = bld * s * (2 + (1 if self.has_z else 0)) + 2 * bln * s
        nread += self.dim * self.N * 4 + (self.dim * 4 if self.has_D else 0)
        nread += self.dim * 4 if self.has_bias else 0
        nwrite = bld * s + self.batch * self.dim * self.N * 4
        return nread + nwrite

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads: shapes, state size, io precision, A pattern, step range and which optional
# operands are present.
WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", "s6-fwd fp32 b1 L256 D64 N16", 1, 256, 64, 16, "f32", "neg_n1",
                     (1e-3, 0.1), has_z=False, has_D=True, seed_index=0),
    "fp32": Workload("fp32", "s6-fwd fp32 b8 L2048 D1536 N16 (d_model 768, expand 2)", 8, 2048,
                     1536, 16, "f32", "neg_n1", (1e-3, 0.1), has_z=True, has_D=True,
                     seed_index=1),
    "bf16": Workload("bf16", "s6-fwd bf16 b16 L4096 D2048 N16 (d_model 1024, expand 2)", 16,
                     4096, 2048, 16, "bf16", "neg_exp_u", (1e-3, 0.1), has_z=True, has_D=True,
                     seed_index=2),
    "long": Workload("long", "s6-fwd bf16 b1 L1048576 D1536 N16 (long sequence)", 1, 1 << 20,
                     1536, 16, "bf16", "neg_n1", (1e-4, 1e-2), has_z=False, has_D=False,
                     seed_index=3),
    "wide": Workload("wide", "s6-fwd bf16 b4 L8192 D5120 N16 (d_model 2560, expand 2)", 4, 8192,
                     5120, 16, "bf16", "neg_n1", (1e-3, 0.1), has_z=True, has_D=True,
                     seed_index=4),
}

BASE_SEED = 0x5153CA00


def _gen(seed: int, name: str, device) -> torch.Generator:
    h = hashlib.sha256(f"{seed}:{name}".encode()).digest()
    g = torch.Generator(device=device)
    g.manual_seed(int.from_bytes(h[:8], "little") & ((1 << 63) - 1))
    return g


def _normal(shape, seed, name, device, chunk: int = 1 << 28) -> torch.Tensor:
    """N(0,1) fp32 draw; very large tensors are drawn in slabs to bound temporary memory."""
    g = _gen(seed, name, device)
    numel = math.prod(shape)
    if numel <= chunk:
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    out = torch.empty(numel, device=device, dtype=torch.float32)
    for i in range(0, numel, chunk):
        n = min(chunk, numel - i)
        out[i:i + n] = torch.randn(n, generator=g, device=device, dtype=torch.float32)
    return out.view(shape)


def _uniform(shape, seed, name, device) -> torch.Tensor:
    g = _gen(seed, name, device)
    return torch.rand(shape, generator=g, device=device, dtype=torch.float64)


def make_inputs(w: Workload, seed: Optional[int] = None, device="cpu") -> Dict[str, torch.Tensor]:
    """Draw every operand of workload ``w``. Returns a dict with u, delta, A, B, C and, when the
    workload has them, z, D (the skip vector) and delta_bias. io tensors are float32 or bfloat16;
    A, D and delta_bias are float32."""
    seed = BASE_SEED + w.seed_index if seed is None else seed
    io_dtype = torch.float32 if w.io == "f32" else torch.bfloat16
    bld = (w.batch, w.L, w.dim)
    bln = (w.batch, w.L, w.N)

    def io_tensor(shape, name):
        x = _normal(shape, seed, name, device)
        return x if io_dtype == torch.float32 else x.to(io_dtype)

    out = {
        "u": io_tensor(bld, "u"),
        "delta": io_tensor(bld, "delta_raw"),
        "B": io_tensor(bln, "B"),
        "C": io_tensor(bln, "C"),
    }
    if w.A_kind == "neg_n1":
        A = -torch.arange(1, w.N + 1, dtype=torch.float32, device=device).repeat(w.dim, 1)
    elif w.A_kind == "neg_exp_u":
        r = _uniform((w.dim, w.N), seed, "A", device)
        A = (-torch.exp(r * math.log(16.0))).to(torch.float32)
    else:
        raise ValueError(w.A_kind)
    out["A"] = A.contiguous()
    if w.has_bias:
        lo, hi = w.dt_range
        r = _uniform((w.dim,), seed, "dt0", device)
        dt0 = torch.exp(math.log(lo) + r * (math.log(hi) - math.log(lo)))
        out["delta_bias"] = (dt0 + torch.log(-torch.expm1(-dt0))).to(torch.float32)
    if w.has_D:
        out["D"] = _normal((w.dim,), seed, "Dskip", device)
    if w.has_z:
        out["z"] = io_tensor(bld, "z")
    return out
