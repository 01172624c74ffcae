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
from parity_util import TOL, rel_err

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
