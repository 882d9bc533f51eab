"""Seeded synthetic inputs for the selective scan and the SSD scan.

This module only draws random numbers; it holds none of the scan's arithmetic. The tests
feed the same tensors to the CUDA library and to the fp64 oracle, and the benchmark uses
it for its workloads. Every input is drawn in fp32 and then cast to the I/O dtype; the
cast values are the ground truth for both sides. A, D and the delta bias stay fp32.

Recipe (draw order A, dt0/bias, D, x, delta noise, B, C, z):
  * A = -(1..N) for every channel (Mamba init A_log = log(1..N), A = -exp(A_log)); for the
    SSD scan one scalar per head, A_h = -U[1, 16].
  * delta_raw ~ N(0, 1); the bias is the inverse softplus of dt0 = exp(U[ln 1e-3, ln 1e-1]),
    so softplus(bias) spans the dt_min = 1e-3 .. dt_max = 0.1 range of the Mamba block's
    dt initialisation; one bias per channel (or per head).
  * x, B, C, z ~ N(0, 1); B and C are one (b, L, N) group shared by all channels / heads.
  * D = 1 (the Mamba init) or N(0, 1), per workload.
Seeds are 20261202 + k for workload k; a replica on rank r adds 1000 * r.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

SEED_BASE = 20261202

_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class ScanWorkload:
    """One Mamba-1 selective-scan workload (shapes in the pages' b, L, D, N notation)."""
    name: str
    batch: int
    seqlen: int
    dim: int
    dstate: int
    dtype: str
    d_skip: str = "ones"        # "ones" | "normal" | "none"
    gate: bool = True           # silu(z) gate present
    chunk_len: int = 0          # 0 = let the library choose
    extra: dict = field(default_factory=dict)

    @property
    def units(self) -> int:
        """State updates: one per (batch, step, channel, state)."""
        return self.batch * self.seqlen * self.dim * self.dstate


@dataclass(frozen=True)
class SSDWorkload:
    """One Mamba-2 SSD chunked-scan workload."""
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    chunk: int
    dtype: str
    d_skip: str = "none"
    gate: bool = False


SCAN_WORKLOADS = {
    0: ScanWorkload("tiny-f32 b1 D4 L64 N4", 1, 64, 4, 4, "f32", "ones", True),
    1: ScanWorkload("mamba130m-layer b8 D1536 L2048 N16 bf16", 8, 2048, 1536, 16, "bf16", "ones", True),
    2: ScanWorkload("mamba2.8b-layer b4 D5120 L2048 N16 bf16", 4, 2048, 5120, 16, "bf16", "normal", True),
    3: ScanWorkload("long-seq b1 D2048 L131072 N16 bf16", 1, 131072, 2048, 16, "bf16", "normal", True,
                    chunk_len=2048),
}
SSD_WORKLOAD = SSDWorkload("mamba2-ssd b4 H64 P64 N128 L4096 Q256 bf16", 4, 4096, 64, 64, 128, 256, "bf16")
SSD_WORKLOAD_INDEX = 4


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, g, device, dtype):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)


def _dt_bias(count, g, device):
    lo, hi = math.log(1e-3), math.log(1e-1)
    dt0 = torch.exp(torch.rand(count, generator=g, device=device, dtype=torch.float64) * (hi - lo) + lo)
    return torch.log(torch.expm1(dt0)).to(torch.float32)


def make_scan_inputs(batch, seqlen, dim, dstate, dtype="bf16", seed=SEED_BASE, device="cpu",
                     d_skip="ones", gate=True, A=None):
    """Draw one selective-scan problem. Returns a dict with x, delta, A, B, C, D, z,
    delta_bias (D and z may be None). ``A`` overrides the default -(1..N) rows."""
    dt = _DTYPES[dtype]
    g = _gen(seed, device)
    if A is None:
        row = -torch.exp(torch.log(torch.arange(1, dstate + 1, dtype=torch.float64)))
        A = row.to(torch.float32).repeat(dim, 1).to(device)
    bias = _dt_bias(dim, g, device)
    if d_skip == "ones":
        D = torch.ones(dim, device=device, dtype=torch.float32)
    elif d_skip == "normal":
        D = torch.randn(dim, generator=g, device=device, dtype=torch.float32)
    else:
        D = None
    x = _normal((batch, seqlen, dim), g, device, dt)
    delta = _normal((batch, seqlen, dim), g, device, dt)
    B = _normal((batch, seqlen, dstate), g, device, dt)
    C = _normal((batch, seqlen, dstate), g, device, dt)
    z = _normal((batch, seqlen, dim), g, device, dt) if gate else None
    return dict(x=x, delta=delta, A=A, B=B, C=C, D=D, z=z, delta_bias=bias)


def scan_workload_inputs(k: int, device="cpu", rank: int = 0, seqlen=None, batch=None, dim=None):
    """Inputs of scan workload k (0..3), optionally with a shorter sequence, batch or width."""
    w = SCAN_WORKLOADS[k]
    return make_scan_inputs(batch or w.batch, seqlen or w.seqlen, dim or w.dim, w.dstate, w.dtype,
                            SEED_BASE + k + 1000 * rank, device, w.d_skip, w.gate)


def make_ssd_inputs(batch, seqlen, nheads, headdim, dstate, dtype="bf16", seed=SEED_BASE, device="cpu",
                    d_skip="none", gate=False, ngroups=1):
    """Draw one SSD problem: x (b, L, H, P), delta (b, L, H), A (H), B, C (b, L, G, N),
    D (H) or None, z (b, L, H, P) or None, delta_bias (H)."""
    dt = _DTYPES[dtype]
    g = _gen(seed, device)
    A = -(torch.rand(nheads, generator=g, device=device, dtype=torch.float32) * 15.0 + 1.0)
    bias = _dt_bias(nheads, g, device)
    if d_skip == "ones":
        D = torch.ones(nheads, device=device, dtype=torch.float32)
    elif d_skip == "normal":
        D = torch.randn(nheads, generator=g, device=device, dtype=torch.float32)
    else:
        D = None
    x = _normal((batch, seqlen, nheads, headdim), g, device, dt)
    delta = _normal((batch, seqlen, nheads), g, device, dt)
    B = _normal((batch, seqlen, ngroups, dstate), g, device, dt)
    C = _normal((batch, seqlen, ngroups, dstate), g, device, dt)
    z = _normal((batch, seqlen, nheads, headdim), g, device, dt) if gate else None
    return dict(x=x, delta=delta, A=A, B=B, C=C, D=D, z=z, delta_bias=bias)


def ssd_workload_inputs(device="cpu", rank: int = 0, seqlen=None, batch=None, nheads=None):
    """Inputs of the SSD workload, optionally with a shorter sequence, batch or head count."""
    w = SSD_WORKLOAD
    return make_ssd_inputs(batch or w.batch, seqlen or w.seqlen, nheads or w.nheads, w.headdim, w.dstate,
                           w.dtype, SEED_BASE + SSD_WORKLOAD_INDEX + 1000 * rank, device, w.d_skip, w.gate)
