"""Python binding of the SSD forward scan library (libssd.so, sm_103a).

Argument marshalling only: tensors are checked for dtype/layout, outputs and
the workspace are allocated with torch on the current CUDA stream, and the
C-ABI entry points of include/ssd.h are called through ctypes.  Every step of
the scan runs in the library's CUDA kernels; there is no CPU fallback, and
importing this package fails loudly if libssd.so has not been built.

    y, final_states = ssd_scan(x, dt, A, B, C, D=None, chunk_size=256,
                               initial_states=None, cu_seqlens=None,
                               return_final_states=True)

computes, for every head h (B/C group g = h // (H // G)),
h_t = exp(dt_t A_h) h_{t-1} + dt_t x_t (outer) B_t and y_t = h_t C_t + D_h x_t,
with the state reset at every cu_seqlens boundary.  Shapes: x (b, L, H, P),
dt (b, L, H) fp32, A (H,) fp32, B/C (b, L, G, N), D (H,) fp32,
initial/final states (nseq, H, P, N) fp32, cu_seqlens (nseq+1,) int32.

If x lives on the CPU, every input is copied to the current CUDA device
(pinned host memory makes the copies asynchronous), the scan runs there and
y / final_states are copied back to the host.

Optional step-size transform (``dt_bias``, ``dt_softplus``, ``dt_limit``):
dt' = clamp(softplus(dt + bias)) applied by the kernels as they read dt.

    y = ssd_step(x, dt, A, B, C, D, state)

is one decode step (one token per sequence; x (b, H, P), dt (b, H), B/C
(b, G, N), state (b, H, P, N) fp32 updated in place).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssd.so")

SSD_F32, SSD_BF16 = 0, 1
ALGOS = {"auto": 0, "simt": 1, "tc": 2, "tc2": 3}
STATUS = {0: "SSD_OK", 1: "SSD_ERR_INVALID_ARG", 2: "SSD_ERR_UNSUPPORTED",
          3: "SSD_ERR_WORKSPACE", 4: "SSD_ERR_CUDA", 5: "SSD_ERR_DEVICE_TIMEOUT",
          6: "SSD_ERR_DEVICE_INPUT"}


class SsdShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64),
                ("nheads", ctypes.c_int32), ("headdim", ctypes.c_int32),
                ("dstate", ctypes.c_int32), ("ngroups", ctypes.c_int32),
                ("chunk_size", ctypes.c_int32), ("nseq", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("algo", ctypes.c_int32)]


class SsdDtTransform(ctypes.Structure):
    _fields_ = [("bias", ctypes.c_void_p), ("softplus", ctypes.c_int32),
                ("dt_min", ctypes.c_float), ("dt_max", ctypes.c_float)]


class SsdStepShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("nheads", ctypes.c_int32),
                ("headdim", ctypes.c_int32), ("dstate", ctypes.c_int32),
                ("ngroups", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class SsdError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


_lib = None


def load_library() -> ctypes.CDLL:
    """Load libssd.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libssd.so not found at {LIB_PATH}; build it with "
                          "`python -m mamba_ssd_layer_03_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    sp = ctypes.POINTER(SsdShape)
    lib.ssd_scan_workspace_size.argtypes = [sp, ctypes.POINTER(sz)]
    lib.ssd_scan_workspace_size.restype = ctypes.c_int
    lib.ssd_scan.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.ssd_scan.restype = ctypes.c_int
    lib.ssd_check_device_status.argtypes = [vp, vp]
    lib.ssd_check_device_status.restype = ctypes.c_int
    lib.ssd_status_string.argtypes = [ctypes.c_int]
    lib.ssd_status_string.restype = ctypes.c_char_p
    lib.ssd_resolve_algo.argtypes = [sp]
    lib.ssd_resolve_algo.restype = ctypes.c_int
    lib.ssd_scan_noalloc.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.ssd_scan_noalloc.restype = ctypes.c_int
    tp = ctypes.POINTER(SsdDtTransform)
    lib.ssd_scan_ex_workspace_size.argtypes = [sp, tp, ctypes.POINTER(sz)]
    lib.ssd_scan_ex_workspace_size.restype = ctypes.c_int
    lib.ssd_scan_ex.argtypes = [sp, vp, vp, tp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.ssd_scan_ex.restype = ctypes.c_int
    lib.ssd_scan_states.argtypes = [sp, vp, vp, tp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.ssd_scan_states.restype = ctypes.c_int
    lib.ssd_step.argtypes = [ctypes.POINTER(SsdStepShape), vp, vp, tp, vp, vp, vp, vp, vp, vp, vp]
    lib.ssd_step.restype = ctypes.c_int
    lib.ssd_selftest_wait_timeout.argtypes = [ctypes.c_int, vp, vp]
    lib.ssd_selftest_wait_timeout.restype = ctypes.c_int
    lib.ssd_seqpar_logdec.argtypes = [sp, vp, tp, vp, vp, vp]
    lib.ssd_seqpar_logdec.restype = ctypes.c_int
    i32 = ctypes.c_int32
    lib.ssd_seqpar_fold.argtypes = [i32, i32, ctypes.c_int64, i32, i32, i32, vp, vp, vp, vp, vp,
                                    vp]
    lib.ssd_seqpar_fold.restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().ssd_status_string(int(code)).decode()


def make_shape(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, nseq,
               dtype: torch.dtype, algo: str = "auto") -> SsdShape:
    if dtype == torch.float32:
        d = SSD_F32
    elif dtype == torch.bfloat16:
        d = SSD_BF16
    else:
        raise TypeError(f"x/B/C dtype must be float32 or bfloat16, got {dtype}")
    return SsdShape(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, nseq, d,
                    ALGOS[algo])


def make_dt_transform(dt_bias: Optional[torch.Tensor] = None, dt_softplus: bool = False,
                      dt_limit=None) -> Optional[SsdDtTransform]:
    """The C struct for a step-size transform, or None when no part is asked
    for.  dt_limit = (dt_min, dt_max); None means no clamp."""
    if dt_bias is None and not dt_softplus and dt_limit is None:
        return None
    lo, hi = (0.0, float("inf")) if dt_limit is None else (float(dt_limit[0]), float(dt_limit[1]))
    return SsdDtTransform(None if dt_bias is None else dt_bias.data_ptr(), 1 if dt_softplus else 0,
                          lo, hi)


def workspace_size(shape: SsdShape, dt_transform: Optional[SsdDtTransform] = None) -> int:
    n = ctypes.c_size_t(0)
    rc = load_library().ssd_scan_ex_workspace_size(
        ctypes.byref(shape), None if dt_transform is None else ctypes.byref(dt_transform),
        ctypes.byref(n))
    if rc != 0:
        raise SsdError(rc, "ssd_scan_workspace_size")
    return int(n.value)


def resolve_algo(shape: SsdShape) -> str:
    rc = load_library().ssd_resolve_algo(ctypes.byref(shape))
    if rc < 0:
        raise SsdError(-rc, "ssd_resolve_algo")
    return {1: "simt", 2: "tc", 3: "tc2"}[rc]


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name, dtype, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def ssd_scan(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
             C: torch.Tensor, D: Optional[torch.Tensor] = None, chunk_size: int = 256,
             initial_states: Optional[torch.Tensor] = None,
             cu_seqlens: Optional[torch.Tensor] = None, return_final_states: bool = True,
             algo: str = "auto", out: Optional[torch.Tensor] = None,
             final_out: Optional[torch.Tensor] = None,
             workspace: Optional[torch.Tensor] = None, check_status: bool = False,
             dt_bias: Optional[torch.Tensor] = None, dt_softplus: bool = False,
             dt_limit=None):
    """Run the SSD forward scan.  Returns (y, final_states or None).

    ``check_status=True`` synchronises and raises if the device reported a
    malformed cu_seqlens or a timed-out wait.  ``out``/``final_out``/
    ``workspace`` let a caller reuse buffers (e.g. inside a timing loop).
    ``dt_bias`` (H,) fp32, ``dt_softplus`` and ``dt_limit`` = (lo, hi) turn
    on the step-size transform dt' = clamp(softplus(dt + bias)).
    """
    if x.device.type == "cpu":
        return _scan_from_host(x, dt, A, B, C, D, chunk_size, initial_states, cu_seqlens,
                               return_final_states, algo, dt_bias, dt_softplus, dt_limit)
    lib = load_library()
    dev = x.device
    if x.dim() != 4:
        raise ValueError("x must be (batch, seqlen, nheads, headdim)")
    b, L, H, P = x.shape
    if B.dim() != 4:
        raise ValueError("B must be (batch, seqlen, ngroups, dstate)")
    G, N = B.shape[2], B.shape[3]
    _check(x, "x", x.dtype, device=dev)
    _check(dt, "dt", torch.float32, (b, L, H), dev)
    _check(A, "A", torch.float32, (H,), dev)
    _check(B, "B", x.dtype, (b, L, G, N), dev)
    _check(C, "C", x.dtype, (b, L, G, N), dev)
    if D is not None:
        _check(D, "D", torch.float32, (H,), dev)
    nseq = b
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int32, device=dev)
        nseq = cu_seqlens.numel() - 1
    if initial_states is not None:
        _check(initial_states, "initial_states", torch.float32, (nseq, H, P, N), dev)
    if dt_bias is not None:
        _check(dt_bias, "dt_bias", torch.float32, (H,), dev)
    tf = make_dt_transform(dt_bias, dt_softplus, dt_limit)
    shape = make_shape(b, L, H, P, N, G, chunk_size, nseq, x.dtype, algo)
    nbytes = workspace_size(shape, tf)
    # caller-supplied buffers are checked like the inputs: the kernels write
    # exactly the documented extents
    if workspace is not None:
        _check(workspace, "workspace", torch.uint8, device=dev)
    if workspace is None or workspace.numel() < nbytes:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    if out is not None:
        _check(out, "out", x.dtype, tuple(x.shape), dev)
    y = out if out is not None else torch.empty_like(x)
    fin = None
    if return_final_states:
        if final_out is not None:
            _check(final_out, "final_out", torch.float32, (nseq, H, P, N), dev)
        fin = final_out if final_out is not None else torch.empty(
            (nseq, H, P, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    if tf is None:
        rc = lib.ssd_scan(ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                          _ptr(D), _ptr(initial_states), _ptr(cu_seqlens), _ptr(y), _ptr(fin),
                          _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                          ctypes.c_void_p(stream))
    else:
        rc = lib.ssd_scan_ex(ctypes.byref(shape), _ptr(x), _ptr(dt), ctypes.byref(tf), _ptr(A),
                             _ptr(B), _ptr(C), _ptr(D), _ptr(initial_states), _ptr(cu_seqlens),
                             _ptr(y), _ptr(fin), _ptr(workspace),
                             ctypes.c_size_t(workspace.numel()), ctypes.c_void_p(stream))
    if rc != 0:
        raise SsdError(rc, "ssd_scan")
    if check_status:
        rc = lib.ssd_check_device_status(_ptr(workspace), ctypes.c_void_p(stream))
        if rc != 0:
            raise SsdError(rc, "ssd_scan (device)")
    return y, fin


def ssd_scan_states(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                    chunk_size: int = 256, initial_states: Optional[torch.Tensor] = None,
                    cu_seqlens: Optional[torch.Tensor] = None, algo: str = "auto",
                    final_out: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None, check_status: bool = False,
                    dt_bias: Optional[torch.Tensor] = None, dt_softplus: bool = False,
                    dt_limit=None) -> torch.Tensor:
    """Final states only (``ssd_scan_states``): what ``ssd_scan`` returns as
    final_states, without computing y.  CUDA tensors; the shape must be one
    the fused tensor-core kernel takes (bf16, headdim 64, dstate 128 or 256),
    else SsdError(SSD_ERR_UNSUPPORTED).  Returns (nseq, H, P, N) fp32."""
    lib = load_library()
    if not isinstance(x, torch.Tensor) or x.dim() != 4:
        raise ValueError("x must be a (batch, seqlen, nheads, headdim) tensor")
    if not isinstance(B, torch.Tensor) or B.dim() != 4:
        raise ValueError("B must be a (batch, seqlen, ngroups, dstate) tensor")
    dev = x.device
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    _check(x, "x", x.dtype, device=dev)
    _check(dt, "dt", torch.float32, (b, L, H), dev)
    _check(A, "A", torch.float32, (H,), dev)
    _check(B, "B", x.dtype, (b, L, G, N), dev)
    nseq = b
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int32, device=dev)
        nseq = cu_seqlens.numel() - 1
    if initial_states is not None:
        _check(initial_states, "initial_states", torch.float32, (nseq, H, P, N), dev)
    if dt_bias is not None:
        _check(dt_bias, "dt_bias", torch.float32, (H,), dev)
    if final_out is not None:
        _check(final_out, "final_out", torch.float32, (nseq, H, P, N), dev)
    if workspace is not None:
        _check(workspace, "workspace", torch.uint8, device=dev)
    if dev.type != "cuda":
        raise ValueError("ssd_scan_states runs on CUDA tensors")
    tf = make_dt_transform(dt_bias, dt_softplus, dt_limit)
    shape = make_shape(b, L, H, P, N, G, chunk_size, nseq, x.dtype, algo)
    nbytes = workspace_size(shape, tf)
    with torch.cuda.device(dev):
        if workspace is None or workspace.numel() < nbytes:
            workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        fin = final_out if final_out is not None else torch.empty(
            (nseq, H, P, N), dtype=torch.float32, device=dev)
        stream = torch.cuda.current_stream(dev).cuda_stream
        rc = lib.ssd_scan_states(ctypes.byref(shape), _ptr(x), _ptr(dt),
                                 None if tf is None else ctypes.byref(tf), _ptr(A), _ptr(B),
                                 _ptr(initial_states), _ptr(cu_seqlens), _ptr(fin),
                                 _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                                 ctypes.c_void_p(stream))
        if rc != 0:
            raise SsdError(rc, "ssd_scan_states")
        if check_status:
            rc = lib.ssd_check_device_status(_ptr(workspace), ctypes.c_void_p(stream))
            if rc != 0:
                raise SsdError(rc, "ssd_scan_states (device)")
    return fin


def ssd_scan_noalloc(x, dt, A, B, C, D=None, chunk_size=256, initial_states=None,
                     out=None, final_out=None, device_status=None, algo: str = "tc"):
    """Scan on the library's own scratch (no workspace, nothing allocated by
    the library).  For callers that cannot allocate device memory while the
    scan runs; outputs may be passed in (``out``, ``final_out``) so that this
    wrapper allocates nothing either.  ``device_status`` (one int32 on the
    device, optional) receives the call's device status word.  Inputs are
    checked like those of ssd_scan(), and the call runs with x's device
    current (the library picks that device's scratch).  ``algo`` is "tc",
    "tc2" or "auto": all three run the two-pass tensor-core kernels.
    Returns (y, final_states or None)."""
    lib = load_library()
    if not isinstance(x, torch.Tensor) or x.dim() != 4:
        raise ValueError("x must be a (batch, seqlen, nheads, headdim) tensor")
    if not isinstance(B, torch.Tensor) or B.dim() != 4:
        raise ValueError("B must be a (batch, seqlen, ngroups, dstate) tensor")
    dev = x.device
    if algo not in ("tc", "tc2", "auto"):
        raise ValueError("ssd_scan_noalloc runs the two-pass tensor-core kernels: "
                         "algo must be 'tc', 'tc2' or 'auto'")
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    _check(x, "x", x.dtype, device=dev)
    _check(dt, "dt", torch.float32, (b, L, H), dev)
    _check(A, "A", torch.float32, (H,), dev)
    _check(B, "B", x.dtype, (b, L, G, N), dev)
    _check(C, "C", x.dtype, (b, L, G, N), dev)
    if D is not None:
        _check(D, "D", torch.float32, (H,), dev)
    if initial_states is not None:
        _check(initial_states, "initial_states", torch.float32, (b, H, P, N), dev)
    if out is not None:
        _check(out, "out", x.dtype, tuple(x.shape), dev)
    if final_out is not None:
        _check(final_out, "final_out", torch.float32, (b, H, P, N), dev)
    if device_status is not None:
        _check(device_status, "device_status", torch.int32, (1,), dev)
    if dev.type != "cuda":
        raise ValueError("ssd_scan_noalloc runs on CUDA tensors")
    shape = make_shape(b, L, H, P, N, G, chunk_size, b, x.dtype, algo)
    with torch.cuda.device(dev):
        y = out if out is not None else torch.empty_like(x)
        stream = torch.cuda.current_stream(dev).cuda_stream
        rc = lib.ssd_scan_noalloc(ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(A), _ptr(B),
                                  _ptr(C), _ptr(D), _ptr(initial_states), _ptr(y),
                                  _ptr(final_out), _ptr(device_status), ctypes.c_void_p(stream))
    if rc != 0:
        raise SsdError(rc, "ssd_scan_noalloc")
    return y, final_out


def ssd_step(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
             C: torch.Tensor, D: Optional[torch.Tensor], state: torch.Tensor,
             dt_bias: Optional[torch.Tensor] = None, dt_softplus: bool = False, dt_limit=None,
             out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One decode step: state (b, H, P, N) fp32 is updated in place; returns
    y (b, H, P).  x (b, H, P) and B, C (b, G, N) in fp32 or bf16, dt (b, H)."""
    lib = load_library()
    if x.dim() != 3 or B.dim() != 3:
        raise ValueError("x must be (batch, nheads, headdim) and B, C (batch, ngroups, dstate)")
    b, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("ssd_step runs on CUDA tensors")
    _check(x, "x", x.dtype, device=dev)
    _check(dt, "dt", torch.float32, (b, H), dev)
    _check(A, "A", torch.float32, (H,), dev)
    _check(B, "B", x.dtype, (b, G, N), dev)
    _check(C, "C", x.dtype, (b, G, N), dev)
    if D is not None:
        _check(D, "D", torch.float32, (H,), dev)
    _check(state, "state", torch.float32, (b, H, P, N), dev)
    if dt_bias is not None:
        _check(dt_bias, "dt_bias", torch.float32, (H,), dev)
    if x.dtype == torch.float32:
        dtype = SSD_F32
    elif x.dtype == torch.bfloat16:
        dtype = SSD_BF16
    else:
        raise TypeError(f"x/B/C dtype must be float32 or bfloat16, got {x.dtype}")
    shape = SsdStepShape(b, H, P, N, G, dtype, 0)
    tf = make_dt_transform(dt_bias, dt_softplus, dt_limit)
    if out is not None:
        _check(out, "out", x.dtype, (b, H, P), dev)
    y = out if out is not None else torch.empty_like(x)
    stream = torch.cuda.current_stream(dev).cuda_stream
    rc = lib.ssd_step(ctypes.byref(shape), _ptr(x), _ptr(dt),
                      None if tf is None else ctypes.byref(tf), _ptr(A), _ptr(B), _ptr(C),
                      _ptr(D), _ptr(state), _ptr(y), ctypes.c_void_p(stream))
    if rc != 0:
        raise SsdError(rc, "ssd_step")
    return y


def selftest_wait_timeout(which: int) -> int:
    """Make one of the kernels' bounded waits run out on purpose (0: an
    mbarrier nothing completes, 1: a handoff flag nothing sets) and return the
    status the device recorded (5, SSD_ERR_DEVICE_TIMEOUT, when the failure
    path works).  Takes about 2 s."""
    words = torch.zeros(2, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    return int(load_library().ssd_selftest_wait_timeout(int(which), _ptr(words),
                                                        ctypes.c_void_p(stream)))


def _scan_from_host(x, dt, A, B, C, D, chunk_size, initial_states, cu_seqlens,
                    return_final_states, algo, dt_bias=None, dt_softplus=False, dt_limit=None):
    dev = torch.device("cuda", torch.cuda.current_device())

    def up(t):
        return None if t is None else t.to(dev, non_blocking=True)

    y, fin = ssd_scan(up(x), up(dt), up(A), up(B), up(C), up(D), chunk_size,
                      up(initial_states), up(cu_seqlens), return_final_states, algo,
                      dt_bias=up(dt_bias), dt_softplus=dt_softplus, dt_limit=dt_limit)
    pin = x.is_pinned()
    y_h = torch.empty(y.shape, dtype=y.dtype, pin_memory=pin)
    y_h.copy_(y, non_blocking=pin)
    fin_h = None
    if fin is not None:
        fin_h = torch.empty(fin.shape, dtype=fin.dtype, pin_memory=pin)
        fin_h.copy_(fin, non_blocking=pin)
    torch.cuda.current_stream(dev).synchronize()
    return y_h, fin_h
