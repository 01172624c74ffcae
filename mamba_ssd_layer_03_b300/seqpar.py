"""Sequence parallelism for the SSD forward scan: one carry exchange per call.

QbitAI article "新架构Mamba更新二代！", section "Mamba-2：更强学习能力，更快训练推理":
sequence parallelism scales the layer to longer sequences.  Every batch row
(sequence) is cut into consecutive shards, shard r on rank r of a process
group (one GPU per rank).  The state is the only quantity that crosses a cut,
so the ranks exchange it once:

1. each rank scans its shard's states from a zero state (``ssd_scan_states``
   where the fused kernel takes the shape: no y is computed; else
   ``ssd_scan``), giving the state S_r its shard leaves, and sums its
   shard's log-decay logdec_r[s, h] = sum_t dt'_t A_h (``ssd_seqpar_logdec``);
2. the ranks all-gather (S_r, logdec_r): H P N + 1 fp32 values per
   (sequence, head) and rank, copied into local buffers;
3. each rank folds the gathered carries of the ranks before it into its
   entry state, H_in(r + 1) = exp(logdec_r) H_in(r) + S_r starting from the
   sequence's initial state (``ssd_seqpar_fold``, which also gives the
   sequence's final state H_in(R), the same on every rank);
4. each rank re-scans its shard from H_in(r) (``ssd_scan`` with
   initial_states), which gives its part of y exactly as the unsharded scan.

The cost per rank is one state-only scan and one full scan of its shard, one
log-decay pass, one fold and one all_gather of (H P N + H) x batch x world
fp32.

``ssd_scan_seqpar`` composes these steps through an ``ops`` object with the
device steps (``states``, ``scan``, ``logdec``, ``fold``) and the collective
(``exchange``); the default, ``CudaOps``, calls the library's kernels through
the C ABI and gathers on the tensors' device (NCCL).  Any other object with
the same five methods can stand in, for example to check the composition and
the collective on CPU ranks.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch
import torch.distributed as dist

from . import (SsdError, _check, _ptr, load_library, make_dt_transform, make_shape,
               resolve_algo, ssd_scan, ssd_scan_states)


def shard_logdec(dt: torch.Tensor, A: torch.Tensor, dt_bias: Optional[torch.Tensor] = None,
                 dt_softplus: bool = False, dt_limit=None,
                 out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Per (sequence, head) log-decay of this shard, sum_t dt'[s, t, h] A_h,
    as a (batch, H) fp32 tensor on dt's device (``ssd_seqpar_logdec``).
    dt (batch, L, H) and A (H,) fp32 CUDA tensors; the optional step-size
    transform is the one ``ssd_scan`` takes."""
    lib = load_library()
    if not isinstance(dt, torch.Tensor) or dt.dim() != 3:
        raise ValueError("dt must be a (batch, seqlen, nheads) tensor")
    dev = dt.device
    b, L, H = dt.shape
    _check(dt, "dt", torch.float32, device=dev)
    _check(A, "A", torch.float32, (H,), dev)
    if dt_bias is not None:
        _check(dt_bias, "dt_bias", torch.float32, (H,), dev)
    if out is not None:
        _check(out, "out", torch.float32, (b, H), dev)
    if dev.type != "cuda":
        raise ValueError("shard_logdec runs on CUDA tensors")
    tf = make_dt_transform(dt_bias, dt_softplus, dt_limit)
    # headdim/dstate/ngroups/chunk do not enter the log-decay; any valid values
    shape = make_shape(b, L, H, 1, 1, 1, 64, b, torch.float32, "simt")
    with torch.cuda.device(dev):
        res = out if out is not None else torch.empty((b, H), dtype=torch.float32, device=dev)
        stream = torch.cuda.current_stream(dev).cuda_stream
        rc = lib.ssd_seqpar_logdec(ctypes.byref(shape), _ptr(dt),
                                   None if tf is None else ctypes.byref(tf), _ptr(A), _ptr(res),
                                   ctypes.c_void_p(stream))
    if rc != 0:
        raise SsdError(rc, "ssd_seqpar_logdec")
    return res


def fold_carries(shard_states: torch.Tensor, shard_logdec_all: torch.Tensor, rank: int,
                 initial_states: Optional[torch.Tensor] = None, want_entry: bool = True,
                 want_final: bool = True):
    """Entry state of shard ``rank`` and the sequence's final state from the
    gathered carries (``ssd_seqpar_fold``).  shard_states (R, b, H, P, N) and
    shard_logdec_all (R, b, H) fp32; initial_states (b, H, P, N) or None.
    Returns (entry or None, final or None)."""
    lib = load_library()
    if not isinstance(shard_states, torch.Tensor) or shard_states.dim() != 5:
        raise ValueError("shard_states must be (nshards, batch, nheads, headdim, dstate)")
    dev = shard_states.device
    R, b, H, P, N = shard_states.shape
    _check(shard_states, "shard_states", torch.float32, device=dev)
    _check(shard_logdec_all, "shard_logdec_all", torch.float32, (R, b, H), dev)
    if initial_states is not None:
        _check(initial_states, "initial_states", torch.float32, (b, H, P, N), dev)
    if not 0 <= rank < R:
        raise ValueError(f"rank {rank} outside [0, {R})")
    if not (want_entry or want_final):
        raise ValueError("ask for the entry state, the final state or both")
    if dev.type != "cuda":
        raise ValueError("fold_carries runs on CUDA tensors")
    with torch.cuda.device(dev):
        entry = torch.empty((b, H, P, N), dtype=torch.float32, device=dev) if want_entry else None
        final = torch.empty((b, H, P, N), dtype=torch.float32, device=dev) if want_final else None
        stream = torch.cuda.current_stream(dev).cuda_stream
        rc = lib.ssd_seqpar_fold(R, rank, b, H, P, N, _ptr(shard_states), _ptr(shard_logdec_all),
                                 _ptr(initial_states), _ptr(entry), _ptr(final),
                                 ctypes.c_void_p(stream))
    if rc != 0:
        raise SsdError(rc, "ssd_seqpar_fold")
    return entry, final


class CudaOps:
    """The three device steps of the exchange on the library's kernels, and
    the all-gather on the tensors' device."""

    def __init__(self, algo: str = "auto", dt_bias=None, dt_softplus=False, dt_limit=None):
        self.algo = algo
        self.dt = dict(dt_bias=dt_bias, dt_softplus=dt_softplus, dt_limit=dt_limit)

    def scan(self, x, dt, A, B, C, D, chunk_size, initial_states, out=None, final=True):
        return ssd_scan(x, dt, A, B, C, D, chunk_size, initial_states, None, final, self.algo,
                        out=out, **self.dt)

    def states(self, x, dt, A, B, C, chunk_size):
        """The shard's end state from a zero state: the state-only scan where
        the fused kernel takes the shape, else a full scan's final states."""
        b, L, H, P = x.shape
        shape = make_shape(b, L, H, P, B.shape[3], B.shape[2], chunk_size, b, x.dtype, self.algo)
        if resolve_algo(shape) == "tc":
            return ssd_scan_states(x, dt, A, B, chunk_size, None, None, self.algo, **self.dt)
        return self.scan(x, dt, A, B, C, None, chunk_size, None)[1]

    def logdec(self, dt, A):
        return shard_logdec(dt, A, **self.dt)

    def fold(self, shard_states, shard_logdec_all, rank, initial_states):
        return fold_carries(shard_states, shard_logdec_all, rank, initial_states)

    def exchange(self, S, logdec, group):
        return exchange_carries(S, logdec, group)


def exchange_carries(S: torch.Tensor, logdec: torch.Tensor, group=None):
    """All-gather this rank's carry (S (b, H, P, N), logdec (b, H), fp32) into
    (R, b, H, P, N) and (R, b, H) buffers of its own, ordered by rank in
    ``group``.  One collective per tensor; the results are plain local copies."""
    world = dist.get_world_size(group)
    S_all = torch.empty((world,) + tuple(S.shape), dtype=S.dtype, device=S.device)
    ld_all = torch.empty((world,) + tuple(logdec.shape), dtype=logdec.dtype,
                         device=logdec.device)
    dist.all_gather_into_tensor(S_all.view(-1), S.contiguous().view(-1), group=group)
    dist.all_gather_into_tensor(ld_all.view(-1), logdec.contiguous().view(-1), group=group)
    return S_all, ld_all


def ssd_scan_seqpar(x, dt, A, B, C, D=None, chunk_size: int = 256, initial_states=None,
                    group=None, ops=None):
    """This rank's shard of a sequence-parallel SSD scan.

    x (b, L_r, H, P), dt (b, L_r, H), B/C (b, L_r, G, N) hold tokens of every
    batch row that fall on this rank (rank r of ``group`` holds the r-th
    consecutive piece; pieces may differ in length, and may be empty).  A, D
    and ``initial_states`` (b, H, P, N; the state before each row's first
    token, used by every rank) are the same on every rank.  Returns
    (y_r, final_states): this rank's y, and every row's state after its last
    token (the same on every rank).  Every rank must call it.
    """
    ops = ops if ops is not None else CudaOps()
    rank = dist.get_rank(group)
    # 1. local carry from a zero state
    S = ops.states(x, dt, A, B, C, chunk_size)
    ld = ops.logdec(dt, A)
    # 2. exchange
    S_all, ld_all = ops.exchange(S, ld, group)
    # 3. fold the shards before this one into the entry state
    entry, final = ops.fold(S_all, ld_all, rank, initial_states)
    # 4. the shard's output from its true entry state
    y, _ = ops.scan(x, dt, A, B, C, D, chunk_size, entry, final=False)
    return y, final
