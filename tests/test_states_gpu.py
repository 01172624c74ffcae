"""The state-only scan (ssd_scan_states) against the fp64 oracle.

It writes what ssd_scan writes to final_states, from the fused kernel's
state-only mode (no C, no y).  Checked element by element against the
oracle's recurrence at 2e-2 and against ssd_scan's own final states on the
same inputs, on narrow lanes (dstate 128, two heads per lane), wide lanes
(dstate 256, grouped B), a few long lanes split between CTAs (recorded
partial states, fold, state-only main run), packed sequences, with and
without initial states, and with the step-size transform.
"""
import pytest
import torch

import oracle
import ssd_synth
from parity_util import TOL, rel_err, to_device

pytestmark = pytest.mark.gpu

CASES = [
    # (name, workload index, overrides)
    ("narrow", 1, dict(batch=2, seqlen=1000, nheads=8, init_states=True)),
    ("narrow_no_init", 1, dict(batch=3, seqlen=777, nheads=6, init_states=False)),
    ("wide_grouped", 3, dict(batch=1, seqlen=900, nheads=8, init_states=True)),
    ("split_lanes", 1, dict(batch=1, seqlen=8192, nheads=2, init_states=True)),
    ("split_lanes_wide", 3, dict(batch=1, seqlen=8192, nheads=8, init_states=True)),
    # four heads per B/C group: CTAs in sets of 4 share each range
    ("split_lanes_wide_sets", 3, dict(batch=1, seqlen=4096, nheads=32, init_states=True)),
    ("varlen", 4, dict(seqlen=5000, nheads=4)),
]


@pytest.mark.parametrize("name,wi,kw", CASES, ids=[c[0] for c in CASES])
def test_state_only_scan_matches_oracle(name, wi, kw):
    import mamba_ssd_layer_03_b300 as ssd
    w = ssd_synth.WORKLOADS[wi]
    inp = ssd_synth.make_inputs(w, seed=61, **kw)
    d = to_device(inp)
    fin = ssd.ssd_scan_states(d["x"], d["dt"], d["A"], d["B"], w.chunk, d["initial_states"],
                              d["cu_seqlens"], check_status=True)
    _, f_scan = ssd.ssd_scan(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], w.chunk,
                             d["initial_states"], d["cu_seqlens"], True, "auto",
                             check_status=True)
    torch.cuda.synchronize()
    _, f_ref = oracle.recurrent(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                inp["initial_states"], inp["cu_seqlens"])
    got = fin.cpu().numpy()
    assert rel_err(got, f_ref) <= TOL["bf16"], rel_err(got, f_ref)
    # the same state arithmetic as the full scan's
    assert rel_err(got, f_scan.cpu().numpy()) <= 1e-6


def test_state_only_scan_with_the_step_size_transform():
    import mamba_ssd_layer_03_b300 as ssd
    w = ssd_synth.WORKLOADS[1]
    inp = ssd_synth.make_inputs(w, seed=62, batch=2, seqlen=1000, nheads=8)
    d = to_device(inp)
    bias = inp["dt_bias"].cuda()
    fin = ssd.ssd_scan_states(d["x"], inp["dt_raw"].cuda(), d["A"], d["B"], w.chunk,
                              dt_bias=bias, dt_softplus=True, dt_limit=(1e-3, 0.08),
                              check_status=True)
    torch.cuda.synchronize()
    dt_ref = oracle.dt_transform(inp["dt_raw"], inp["dt_bias"], True, 1e-3, 0.08)
    _, f_ref = oracle.recurrent(inp["x"], dt_ref, inp["A"], inp["B"], inp["C"])
    assert rel_err(fin.cpu().numpy(), f_ref) <= TOL["bf16"]


def test_state_only_scan_refuses_shapes_without_the_fused_kernel():
    import mamba_ssd_layer_03_b300 as ssd
    w = ssd_synth.WORKLOADS[0]      # fp32: SIMT only
    inp = ssd_synth.make_inputs(w, seed=63)
    d = to_device(inp)
    with pytest.raises(ssd.SsdError):
        ssd.ssd_scan_states(d["x"], d["dt"], d["A"], d["B"], w.chunk)


def test_state_only_scan_rejects_bad_arguments_on_host():
    import ctypes
    import mamba_ssd_layer_03_b300 as ssd
    lib = ssd.load_library()
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the checks come first
    ws = ctypes.c_void_p(1 << 24)
    bf = ssd.make_shape(2, 512, 4, 64, 128, 1, 256, 2, torch.bfloat16, "auto")

    def call(shape, final=fake, wsb=1 << 30, x=fake):
        return lib.ssd_scan_states(ctypes.byref(shape), x, fake, None, fake, fake, None, None,
                                   final, ws, ctypes.c_size_t(wsb), None)

    assert call(bf, final=None) == 1
    assert call(bf, x=None) == 1
    assert call(bf, wsb=1024) == 3
    assert call(ssd.make_shape(2, 512, 4, 64, 128, 1, 256, 1, torch.bfloat16, "auto")) == 1
