"""CPU oracle for the SSD forward scan -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA path shares no code with it.

Two independent formulations, both in fp64:

* ``recurrent`` -- the token-by-token selective SSM recurrence, in C
  (``ssd_oracle.c``, built with gcc/OpenMP by ``build()``).  Source: Mamba-1
  walkthrough "Mamba: Linear-Time Sequence Modeling with Selective State
  Spaces", section 三(二) (selective SSM with input-dependent B, C, Delta) and
  section 三 3 (Abar = exp(Delta A)).
* ``quadratic`` -- the same linear map written as multiplication by the
  semiseparable matrix M = L o (C B^T) (QbitAI article "新架构Mamba更新二代！",
  section "统一SSM和注意力机制": an SSM is a semiseparable-matrix transform and
  is equivalent to masked attention whose mask L is semiseparable).  It is
  O(T^2) per (sequence, head) and meant for tiny inputs only.  Every decay
  sum is formed directly as a sum over its own range, never as a difference
  of two cumulative sums.

A third formulation, the algorithm the pages give for evaluating that matrix
product (QbitAI article, section "Mamba-2：更强学习能力，更快训练推理": block
decomposition of the semiseparable matrix into chunk-local masked quadratic
products plus a recurrence between chunks):

* ``chunked`` -- per chunk of ``chunk`` tokens, in the pages' order: the
  cumulative decay within the chunk (``chunk_decay``), the chunk's state
  contribution (``chunk_state``), the state passed from chunk to chunk
  (``state_passing``), and the chunk's output from its masked block and its
  entry state (``chunk_output``).  Chunks restart at every sequence start.

Two helpers around them, also fp64:

* ``dt_transform`` -- the step size Delta = tau_Delta(parameter + s_Delta(x))
  with tau_Delta = softplus (Mamba-1 walkthrough, section 三(二)): a bias per
  head, softplus, then an optional clamp.
* ``step`` -- one decode step, i.e. the recurrence over a single token with
  the given state as the initial state (the recurrent mode used for
  inference: Mamba-1 walkthrough, sections 二(一) and 四(五)).

Readings taken where the pages are silent (one A scalar per head, Bbar = dt B,
y from the updated state, an optional D skip term, contiguous head -> group
mapping, exact state reset at packed-sequence boundaries) are shared by both
formulations because both are written from the same definition.

Parity unpinned: nothing.  Every function here is pinned by the tests in
``tests/test_oracle_pins.py`` against closed forms, hand-computed golden
fixtures, the recurrent/quadratic duality, the chunked form's agreement with
both at every chunk size, and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

# Mutations that tests plant in the oracle (see ssd_oracle.c).
MUTATIONS = {
    "y_from_old_state": 1,
    "decay_sign": 2,
    "group_map": 3,
    "drop_D": 4,
    "drop_dt_input": 5,
    "no_reset": 6,
}


def build(force: bool = False) -> str:
    """Compile ssd_oracle.c into liboracle.so with gcc (-O2 -fopenmp)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
               "-Wall", "-o", _LIB, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        d = ctypes.c_void_p
        i64, i32 = ctypes.c_int64, ctypes.c_int
        lib.ssd_oracle_recurrent.argtypes = [i64, i64, i32, i32, i32, i32, i32,
                                             d, d, d, d, d, d, d, d, d, d, d, i32, i32]
        lib.ssd_oracle_recurrent.restype = i32
        lib.ssd_oracle_recurrent_mut.argtypes = [i64, i64, i32, i32, i32, i32, i32,
                                                 d, d, d, d, d, d, d, d, d, d, i32]
        lib.ssd_oracle_recurrent_mut.restype = i32
        lib.ssd_oracle_max_threads.restype = i32
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().ssd_oracle_max_threads())


def _f64(a) -> Optional[np.ndarray]:
    """Exact upcast of a torch tensor (fp32/bf16) or array to contiguous fp64."""
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().to("cpu")
        import torch
        a = a.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _prep(x, dt, A, B, C, D, initial_states, cu_seqlens):
    x, dt, A, B, C = (_f64(t) for t in (x, dt, A, B, C))
    D = _f64(D)
    init = _f64(initial_states)
    cu = None
    if cu_seqlens is not None:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    nseq = (len(cu) - 1) if cu is not None else b
    return x, dt, A, B, C, D, init, cu, (b, L, H, P, N, G, nseq)


def recurrent(x, dt, A, B, C, D=None, initial_states=None, cu_seqlens=None,
              units: Optional[Sequence[int]] = None, nthreads: int = 0,
              mutation: Optional[str] = None):
    """fp64 token-by-token recurrence.  Returns (y, final_states) as float64.

    ``units`` restricts the work to the listed (sequence * H + head) units;
    rows of y belonging to other units are left as NaN.
    """
    lib = _load()
    x, dt, A, B, C, D, init, cu, (b, L, H, P, N, G, nseq) = _prep(
        x, dt, A, B, C, D, initial_states, cu_seqlens)
    y = np.full((b, L, H, P), np.nan)
    fin = np.full((nseq, H, P, N), np.nan)
    if mutation is not None:
        rc = lib.ssd_oracle_recurrent_mut(b, L, H, P, N, G, nseq, _ptr(cu), _ptr(x), _ptr(dt),
                                          _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init),
                                          _ptr(y), _ptr(fin), MUTATIONS[mutation])
    else:
        uarr = None
        if units is not None:
            uarr = np.ascontiguousarray(np.asarray(list(units), dtype=np.int32))
        rc = lib.ssd_oracle_recurrent(b, L, H, P, N, G, nseq, _ptr(cu), _ptr(x), _ptr(dt),
                                      _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init),
                                      _ptr(y), _ptr(fin), _ptr(uarr),
                                      0 if uarr is None else len(uarr), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return y, fin


def recurrent_unit(x, dt, A, B, C, D, initial_states, cu_seqlens, s: int, h: int):
    """fp64 recurrence of the single (sequence s, head h) unit, from sliced
    inputs (only that unit's tokens, head and group are converted to fp64).
    Returns (y (T, P), final_state (P, N))."""
    H, G = x.shape[2], B.shape[2]
    g = h // (H // G)
    if cu_seqlens is not None:
        row, t0, t1 = 0, int(cu_seqlens[s]), int(cu_seqlens[s + 1])
    else:
        row, t0, t1 = s, 0, x.shape[1]
    sl = lambda t, k: t[row:row + 1, t0:t1, k:k + 1]
    S0 = None if initial_states is None else initial_states[s:s + 1, h:h + 1]
    y, fin = recurrent(sl(x, h), dt[row:row + 1, t0:t1, h:h + 1], A[h:h + 1], sl(B, g), sl(C, g),
                       None if D is None else D[h:h + 1], S0, None, nthreads=1)
    return y[0, :, 0, :], fin[0, 0]


def dt_transform(dt, bias=None, softplus: bool = False, dt_min: float = 0.0,
                 dt_max: float = float("inf")) -> np.ndarray:
    """fp64 step sizes dt' = clamp(softplus(dt + bias[h])) for dt (..., H).
    softplus(z) = log(1 + e^z), evaluated as logaddexp(0, z) so that it
    neither overflows for large z nor loses e^z for very negative z."""
    z = _f64(dt)
    if bias is not None:
        z = z + _f64(bias)
    if softplus:
        z = np.logaddexp(0.0, z)
    return np.minimum(np.maximum(z, dt_min), dt_max)


def step(x, dt, A, B, C, D, state):
    """fp64 decode step of sequences holding one token each: x (b, H, P),
    dt (b, H), B/C (b, G, N), state (b, H, P, N).  Returns (y (b, H, P),
    new state (b, H, P, N)): the recurrence over that single token starting
    from `state`."""
    x, dt, B, C = (_f64(t) for t in (x, dt, B, C))
    y, fin = recurrent(x[:, None], dt[:, None], A, B[:, None], C[:, None], D,
                       initial_states=state)
    return y[:, 0], fin


def quadratic(x, dt, A, B, C, D=None, initial_states=None, cu_seqlens=None):
    """fp64 semiseparable-matrix form, y = (L o (C B^T)) . X + init term + D x.

    For each sequence and head, with a_k = dt_k A_h:
      M[i, j]  = (C_i . B_j) * exp(sum_{k=j+1..i} a_k) * dt_j      (j <= i)
      y_i      = sum_j M[i, j] x_j + exp(sum_{k<=i} a_k) C_i . S0 + D_h x_i
      final    = exp(sum_k a_k) S0 + sum_j exp(sum_{k>j} a_k) dt_j x_j (outer) B_j
    Every exponent is a direct sum over its own index range.
    """
    x, dt, A, B, C, D, init, cu, (b, L, H, P, N, G, nseq) = _prep(
        x, dt, A, B, C, D, initial_states, cu_seqlens)
    y = np.zeros((b, L, H, P))
    fin = np.zeros((nseq, H, P, N))
    hpg = H // G
    for s in range(nseq):
        row = 0 if cu is not None else s
        t0 = int(cu[s]) if cu is not None else 0
        t1 = int(cu[s + 1]) if cu is not None else L
        T = t1 - t0
        for h in range(H):
            g = h // hpg
            a = dt[row, t0:t1, h] * A[h]
            Xs = x[row, t0:t1, h, :]                 # (T, P)
            Bs = B[row, t0:t1, g, :]                 # (T, N)
            Cs = C[row, t0:t1, g, :]
            dts = dt[row, t0:t1, h]
            M = np.zeros((T, T))
            for i in range(T):
                for j in range(i + 1):
                    M[i, j] = float(Cs[i] @ Bs[j]) * np.exp(np.sum(a[j + 1:i + 1])) * dts[j]
            yv = M @ Xs
            S0 = init[s, h] if init is not None else np.zeros((P, N))
            for i in range(T):
                yv[i] += np.exp(np.sum(a[:i + 1])) * (S0 @ Cs[i])
            if D is not None:
                yv += D[h] * Xs
            y[row, t0:t1, h, :] = yv
            F = np.exp(np.sum(a)) * S0
            for j in range(T):
                F = F + np.exp(np.sum(a[j + 1:])) * dts[j] * np.outer(Xs[j], Bs[j])
            fin[s, h] = F
    return y, fin


# ---------------------------------------------------------------- block decomposition
# QbitAI article "新架构Mamba更新二代！", section "Mamba-2：更强学习能力，更快训练推理":
# the semiseparable matrix is cut into chunks; diagonal blocks are masked
# quadratic products, off-diagonal blocks are low rank and pass through a
# per-chunk state.  Notation per (sequence, head): a_k = dt_k A_h, tokens of
# one chunk indexed i, j from 0.


def chunk_decay(a: np.ndarray) -> np.ndarray:
    """Cumulative decay within one chunk: cs_i = a_0 + ... + a_i."""
    return np.cumsum(a)


def chunk_state(Bc: np.ndarray, Xc: np.ndarray, dtc: np.ndarray, cs: np.ndarray) -> np.ndarray:
    """State the chunk's own tokens leave at its end, from a zero entry state:
    S = sum_j exp(cs_last - cs_j) dt_j x_j (outer) B_j, shape (P, N)."""
    w = np.exp(cs[-1] - cs) * dtc                       # (T,)
    return (Xc * w[:, None]).T @ Bc


def state_passing(S: Sequence[np.ndarray], cs_last: Sequence[float], S0: np.ndarray):
    """Entry state of every chunk and the final state:
    H_0 = S0, H_{c+1} = exp(cs_last_c) H_c + S_c."""
    entries = []
    Hc = S0
    for Sc, e in zip(S, cs_last):
        entries.append(Hc)
        Hc = np.exp(e) * Hc + Sc
    return entries, Hc


def chunk_output(Cc, Bc, Xc, dtc, cs, H_entry, Dh) -> np.ndarray:
    """Output of one chunk: y_i = sum_{j<=i} (C_i . B_j) exp(cs_i - cs_j) dt_j x_j
    + exp(cs_i) C_i . H_entry + D_h x_i, shape (T, P)."""
    T = len(cs)
    causal = np.tril(np.ones((T, T), dtype=bool))       # j <= i
    Lmask = np.where(causal, np.exp(np.where(causal, cs[:, None] - cs[None, :], 0.0)), 0.0) * dtc[None, :]
    y = ((Cc @ Bc.T) * Lmask) @ Xc
    y += np.exp(cs)[:, None] * (Cc @ H_entry.T)
    if Dh is not None:
        y += Dh * Xc
    return y


def chunked(x, dt, A, B, C, D=None, initial_states=None, cu_seqlens=None, chunk: int = 64):
    """fp64 block decomposition with chunks of ``chunk`` tokens (the last chunk
    of a sequence may be shorter).  Returns (y, final_states) as float64."""
    if chunk < 1:
        raise ValueError("chunk must be positive")
    x, dt, A, B, C, D, init, cu, (b, L, H, P, N, G, nseq) = _prep(
        x, dt, A, B, C, D, initial_states, cu_seqlens)
    y = np.zeros((b, L, H, P))
    fin = np.zeros((nseq, H, P, N))
    hpg = H // G
    for s in range(nseq):
        row = 0 if cu is not None else s
        t0 = int(cu[s]) if cu is not None else 0
        t1 = int(cu[s + 1]) if cu is not None else L
        for h in range(H):
            g = h // hpg
            S0 = init[s, h] if init is not None else np.zeros((P, N))
            bounds = [(c, min(c + chunk, t1)) for c in range(t0, t1, chunk)]
            parts = []
            for c0, c1 in bounds:
                dtc = dt[row, c0:c1, h]
                cs = chunk_decay(dtc * A[h])
                parts.append((dtc, cs, chunk_state(B[row, c0:c1, g], x[row, c0:c1, h], dtc, cs)))
            entries, fin[s, h] = state_passing([p[2] for p in parts], [p[1][-1] for p in parts], S0)
            for (c0, c1), (dtc, cs, _), He in zip(bounds, parts, entries):
                y[row, c0:c1, h] = chunk_output(C[row, c0:c1, g], B[row, c0:c1, g], x[row, c0:c1, h],
                                                dtc, cs, He, None if D is None else D[h])
    return y, fin
