"""The allocation-free entry point, ssd_scan_noalloc(), through the C ABI.

It serves callers that cannot allocate device memory while they run the scan
(code inside another framework's execution hook, where that framework owns
every device allocation, or a real-time loop that forbids allocation after
start-up).  It must give the same result as ssd_scan() on the same inputs,
call after call, while using only the library's own fixed scratch.  This file
is collected last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import ssd_synth
from parity_util import TOL, oracle_full, rel_err

pytestmark = pytest.mark.gpu


def _dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _noalloc(lib, shape, d, y, fin, status, stream):
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return lib.ssd_scan_noalloc(ctypes.byref(shape), p(d["x"]), p(d["dt"]), p(d["A"]), p(d["B"]),
                                p(d["C"]), p(d["D"]), p(d["initial_states"]), p(y), p(fin),
                                p(status), ctypes.c_void_p(stream))


def test_noalloc_matches_workspace_entry_point_twice():
    import mamba_ssd_layer_03_b300 as ssd
    lib = ssd.load_library()
    w = ssd_synth.WORKLOADS[1]
    inp = ssd_synth.make_inputs(w, seed=21, batch=2, seqlen=1000, nheads=6, init_states=True)
    d = _dev(inp)
    # the allocation-free entry point runs the two-pass tensor-core kernels
    y_ref, f_ref = ssd.ssd_scan(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], w.chunk,
                                d["initial_states"], None, True, "tc2", check_status=True)
    torch.cuda.synchronize()
    shape = ssd.make_shape(inp["batch"], inp["seqlen"], inp["nheads"], inp["headdim"],
                           inp["dstate"], inp["ngroups"], w.chunk, inp["nseq"], torch.bfloat16, "tc")
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        y = torch.full_like(d["x"], float("nan"))
        fin = torch.full_like(f_ref, float("nan"))
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        rc = _noalloc(lib, shape, d, y, fin, status, stream)
        assert rc == 0, ssd.status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert rel_err(y.float().cpu().numpy(), y_ref.float().cpu().numpy()) <= TOL["bf16"], call
        assert rel_err(fin.cpu().numpy(), f_ref.cpu().numpy()) <= TOL["bf16"], call


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import mamba_ssd_layer_03_b300 as ssd
    lib = ssd.load_library()
    # The 2.7B-shaped layer needs far more than the fixed scratch holds.
    w = ssd_synth.WORKLOADS[2]
    need = ssd.make_shape(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk,
                          w.batch, torch.bfloat16, "tc2")
    assert ssd.workspace_size(need) > (32 << 20)
    shape = ssd.make_shape(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk,
                           w.batch, torch.bfloat16, "tc")
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the size check comes first
    rc = lib.ssd_scan_noalloc(ctypes.byref(shape), fake, fake, fake, fake, fake, None, None, fake,
                              None, None, None)
    assert rc == 3, ssd.status_string(rc)


@pytest.mark.parametrize("algo", ["tc", "tc2"])
def test_noalloc_matches_oracle_with_and_without_D(algo):
    """Element by element against the fp64 oracle, with D and with D = 0 (D x
    dominates |y| at these scales and would hide errors in the scan term), for
    both algorithm values the call accepts; two calls in a row each time, so
    that the second runs on scratch the first one left behind."""
    import mamba_ssd_layer_03_b300 as ssd
    lib = ssd.load_library()
    w = ssd_synth.WORKLOADS[3]    # dstate 256, 4 heads per B/C group
    inp = ssd_synth.make_inputs(w, seed=22, batch=2, seqlen=700, nheads=8, init_states=True)
    d = _dev(inp)
    shape = ssd.make_shape(inp["batch"], inp["seqlen"], inp["nheads"], inp["headdim"],
                           inp["dstate"], inp["ngroups"], w.chunk, inp["nseq"], torch.bfloat16, algo)
    stream = torch.cuda.current_stream().cuda_stream
    for with_D in (True, False):
        y_ref, f_ref = oracle_full(inp, D=with_D)
        dd = dict(d)
        if not with_D:
            dd["D"] = None
        for call in range(2):
            y = torch.full_like(d["x"], float("nan"))
            fin = torch.full(f_ref.shape, float("nan"), device="cuda")
            status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
            rc = _noalloc(lib, shape, dd, y, fin, status, stream)
            assert rc == 0, ssd.status_string(rc)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            ey = rel_err(y.float().cpu().numpy(), y_ref)
            ef = rel_err(fin.cpu().numpy(), f_ref)
            assert ey <= TOL["bf16"], (with_D, call, ey)
            assert ef <= TOL["bf16"], (with_D, call, ef)


def test_noalloc_python_wrapper_twice():
    """The Python binding of the call, with its own input checks and the
    inputs' device made current, caller-supplied outputs (so nothing is
    allocated per call), against the oracle on two calls in a row."""
    import mamba_ssd_layer_03_b300 as ssd
    w = ssd_synth.WORKLOADS[1]
    inp = ssd_synth.make_inputs(w, seed=23, batch=1, seqlen=1300, nheads=4, init_states=True)
    d = _dev(inp)
    y_ref, f_ref = oracle_full(inp)
    y = torch.empty_like(d["x"])
    fin = torch.empty(f_ref.shape, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        y.fill_(float("nan"))
        fin.fill_(float("nan"))
        yo, fo = ssd.ssd_scan_noalloc(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], w.chunk,
                                      d["initial_states"], out=y, final_out=fin,
                                      device_status=status)
        torch.cuda.synchronize()
        assert yo is y and fo is fin
        assert int(status.item()) == 0
        assert rel_err(y.float().cpu().numpy(), y_ref) <= TOL["bf16"], call
        assert rel_err(fin.cpu().numpy(), f_ref) <= TOL["bf16"], call
