"""Seeded synthetic inputs for the SSD forward scan.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark.  It only draws random numbers and lays them out; none of the scan's
arithmetic lives here.  The one non-trivial expression, ``dt = softplus(n +
bias)``, is the selection step that sits *upstream* of the scan: the Mamba-1
walkthrough ("Mamba: Linear-Time Sequence Modeling with Selective State
Spaces", section 三(二) "引入选择机制到 SSM 中") puts the softplus activation
tau_Delta on the Delta projection before the recurrence, so the scan receives
dt already positive.

Distributions (the five workload shapes of the Mamba-2 SSD layer):
  x, B, C ~ N(0, 1); B and C scaled by 1/sqrt(N) except in the tiny fp32 case
  dt0_h   = exp(U[ln 1e-3, ln 0.1])            (log-uniform per head)
  bias_h  = dt0_h + ln(-expm1(-dt0_h))         (inverse softplus of dt0_h)
  dt      = softplus(n + bias_h), n ~ N(0, sd 0.5)
  A_h     = -exp(U[ln 1, ln 16]);  D_h ~ N(0, 1)
  initial_states ~ N(0, sd 0.1) (large-state case only)
  varlen: integer segment lengths ~ U{64..4096} drawn until the total reaches
          the token count, the last one truncated.
Draw order from one ``torch.Generator`` seeded with ``seed``: x, B, C,
dt-noise, dt-bias, A, D, initial_states, segment lengths.  Everything is drawn
in fp32 and then cast to the storage dtype.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, asdict
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk: int
    dtype: str                      # "fp32" or "bf16": storage of x, B, C, y
    scale_bc: bool = True           # B, C scaled by 1/sqrt(N)
    init_states: bool = False       # draw nonzero initial_states
    varlen: Optional[tuple] = None  # (min_len, max_len) of packed segments

    def as_dict(self):
        d = asdict(self)
        d["varlen"] = list(self.varlen) if self.varlen else None
        return d


# The five workloads of the SSD layer.  Index 2 is the 2.7B-model-shaped layer
# (d_inner = 80 heads x 64 = 5120) on which throughput is reported.
WORKLOADS = [
    Workload("tiny_fp32", 1, 256, 2, 16, 16, 1, 64, "fp32", scale_bc=False),
    Workload("bf16_b2_L2048_h24", 2, 2048, 24, 64, 128, 1, 256, "bf16"),
    Workload("ssd_2p7b_b4_L8192_h80", 4, 8192, 80, 64, 128, 1, 256, "bf16"),
    Workload("large_state_N256_G8", 2, 16384, 32, 64, 256, 8, 256, "bf16",
             init_states=True),
    Workload("varlen_T32768_h64", 1, 32768, 64, 64, 128, 1, 256, "bf16",
             varlen=(64, 4096)),
]


def storage_dtype(name: str) -> torch.dtype:
    return {"fp32": torch.float32, "bf16": torch.bfloat16}[name]


def make_inputs(w: Workload, seed: int = 0, *, batch: Optional[int] = None,
                seqlen: Optional[int] = None, nheads: Optional[int] = None,
                init_states: Optional[bool] = None,
                segment_lengths: Optional[list] = None) -> dict:
    """Draw one input set for workload ``w`` (CPU tensors, storage dtypes).

    Overrides (batch, seqlen, nheads, init_states, explicit segment lengths)
    keep the distributions and change only the shape; tests use them for
    ragged and degenerate cases.
    Returns a dict with x, dt, A, B, C, D, initial_states (or None),
    cu_seqlens (int32 or None) and the shape scalars, plus the parts dt is
    made of (dt_raw = the noise n, dt_bias = bias_h), for the scan's optional
    step-size transform.
    """
    b = w.batch if batch is None else batch
    L = w.seqlen if seqlen is None else seqlen
    H = w.nheads if nheads is None else nheads
    P, N, G = w.headdim, w.dstate, w.ngroups
    use_init = w.init_states if init_states is None else init_states
    dt_store = storage_dtype(w.dtype)
    g = torch.Generator().manual_seed(seed)

    x = torch.randn(b, L, H, P, generator=g)
    Bm = torch.randn(b, L, G, N, generator=g)
    Cm = torch.randn(b, L, G, N, generator=g)
    if w.scale_bc:
        Bm = Bm / math.sqrt(N)
        Cm = Cm / math.sqrt(N)
    dt_noise = torch.randn(b, L, H, generator=g) * 0.5
    u = torch.rand(H, generator=g)
    dt0 = torch.exp(math.log(1e-3) + u * (math.log(0.1) - math.log(1e-3)))
    bias = dt0 + torch.log(-torch.expm1(-dt0))
    dt = torch.nn.functional.softplus(dt_noise + bias)
    ua = torch.rand(H, generator=g)
    A = -torch.exp(ua * math.log(16.0))
    D = torch.randn(H, generator=g)

    cu = None
    nseq = b
    if w.varlen is not None or segment_lengths is not None:
        if b != 1:
            raise ValueError("packed variable-length input needs batch == 1")
        if segment_lengths is None:
            lo, hi = w.varlen
            segs = []
            total = 0
            while total < L:
                s = int(torch.randint(lo, hi + 1, (1,), generator=g))
                segs.append(s)
                total += s
            segs[-1] -= total - L
        else:
            segs = list(segment_lengths)
            if sum(segs) != L or min(segs) < 0:
                raise ValueError("segment lengths must be >= 0 and sum to seqlen")
        cu = torch.zeros(len(segs) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(segs, dtype=torch.int64), 0).to(torch.int32)
        nseq = len(segs)

    init = None
    if use_init:
        init = torch.randn(nseq, H, P, N, generator=g) * 0.1

    return dict(
        x=x.to(dt_store).contiguous(), dt=dt.float().contiguous(),
        A=A.float().contiguous(), B=Bm.to(dt_store).contiguous(),
        C=Cm.to(dt_store).contiguous(), D=D.float().contiguous(),
        initial_states=None if init is None else init.float().contiguous(),
        cu_seqlens=cu, batch=b, seqlen=L, nheads=H, headdim=P, dstate=N,
        ngroups=G, chunk=w.chunk, nseq=nseq, dtype=w.dtype,
        dt_raw=dt_noise.float().contiguous(), dt_bias=bias.float().contiguous())


def make_dt_parts(w: Workload, seed: int = 0, **shape):
    """(dt_raw, dt_bias, dt) of the input set make_inputs(w, seed, **shape)
    draws: dt = softplus(dt_raw + dt_bias[h])."""
    inp = make_inputs(w, seed, **shape)
    return inp["dt_raw"], inp["dt_bias"], inp["dt"]
