"""GPU parity of the decode step (ssd_step) and of the scan with the step-size
transform (ssd_scan_ex), element by element against the fp64 oracle.

The decode step is the recurrent form over one token per sequence with the
state updated in place; the oracle is its recurrence over that token
(oracle.step).  The transform dt' = clamp(softplus(dt + bias)) is checked
through every scan path (fused, two-pass, SIMT) and through the step, against
oracle.dt_transform followed by the oracle's recurrence.
"""
import numpy as np
import pytest
import torch

import oracle
import ssd_synth
from parity_util import TOL, rel_err

pytestmark = pytest.mark.gpu


def _step_inputs(seed, b, H, P, N, G, dtype):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(b, H, P, generator=g)
    Bm = torch.randn(b, G, N, generator=g) / np.sqrt(N)
    Cm = torch.randn(b, G, N, generator=g) / np.sqrt(N)
    raw = torch.randn(b, H, generator=g) * 0.5
    dt0 = torch.exp(np.log(1e-3) + torch.rand(H, generator=g) * (np.log(0.1) - np.log(1e-3)))
    bias = dt0 + torch.log(-torch.expm1(-dt0))
    A = -torch.exp(torch.rand(H, generator=g) * np.log(16.0))
    D = torch.randn(H, generator=g)
    S = torch.randn(b, H, P, N, generator=g) * 0.3
    st = dtype
    return dict(x=x.to(st), B=Bm.to(st), C=Cm.to(st), raw=raw, bias=bias,
                dt=torch.nn.functional.softplus(raw + bias), A=A, D=D, S=S)


def _run_step(inp, D=True, **tf):
    import mamba_ssd_layer_03_b300 as ssd
    c = {k: v.cuda() for k, v in inp.items()}
    S = c["S"].clone()
    dt = c["raw"] if tf else c["dt"]
    if tf.get("dt_bias") is not None:
        tf = dict(tf, dt_bias=c["bias"])
    y = ssd.ssd_step(c["x"], dt, c["A"], c["B"], c["C"], c["D"] if D else None, S, **tf)
    torch.cuda.synchronize()
    return y.float().cpu().numpy(), S.cpu().numpy()


STEP_CASES = [
    # (b, H, P, N, G, dtype)
    (3, 4, 16, 16, 2, torch.float32),
    (2, 6, 64, 128, 1, torch.float32),
    (4, 8, 64, 128, 1, torch.bfloat16),
    (2, 32, 64, 256, 8, torch.bfloat16),
    (3, 5, 24, 37, 5, torch.float32),      # dstate not a multiple of 4: scalar path
    (1, 2, 200, 1024, 1, torch.bfloat16),  # the largest state the step takes
]


@pytest.mark.parametrize("case", STEP_CASES, ids=lambda c: f"b{c[0]}h{c[1]}p{c[2]}n{c[3]}g{c[4]}-{str(c[5])[6:]}")
@pytest.mark.parametrize("D", [True, False])
def test_step_matches_oracle(case, D):
    b, H, P, N, G, dt = case
    inp = _step_inputs(1, b, H, P, N, G, dt)
    y, S = _run_step(inp, D=D)
    y_ref, S_ref = oracle.step(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                               inp["D"] if D else None, inp["S"])
    tol = TOL["fp32"] if dt == torch.float32 else TOL["bf16"]
    assert rel_err(y, y_ref) <= tol
    # the state is fp32 arithmetic on the given inputs: fp32 tolerance
    assert rel_err(S, S_ref) <= TOL["fp32"]


def test_step_sequence_equals_scan():
    """Twelve decode steps in a row give the scan's outputs token by token and
    its final state."""
    import mamba_ssd_layer_03_b300 as ssd
    w = ssd_synth.WORKLOADS[1]
    inp = ssd_synth.make_inputs(w, seed=4, batch=2, seqlen=12, nheads=4, init_states=True)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    S = d["initial_states"].clone()
    ys = []
    for t in range(12):
        y = ssd.ssd_step(d["x"][:, t].contiguous(), d["dt"][:, t].contiguous(), d["A"],
                         d["B"][:, t].contiguous(), d["C"][:, t].contiguous(), d["D"], S)
        ys.append(y.float().cpu().numpy())
    torch.cuda.synchronize()
    y_ref, fin_ref = oracle.recurrent(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                                      inp["D"], inp["initial_states"])
    assert rel_err(np.stack(ys, axis=1), y_ref) <= TOL["bf16"]
    assert rel_err(S.cpu().numpy(), fin_ref) <= TOL["fp32"]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("limit", [None, (0.004, 0.05)])
def test_step_with_dt_transform(dtype, limit):
    inp = _step_inputs(7, 3, 8, 64, 128, 2, dtype)
    y, S = _run_step(inp, dt_bias=True, dt_softplus=True, dt_limit=limit)
    lo, hi = (0.0, np.inf) if limit is None else limit
    dtp = oracle.dt_transform(inp["raw"], bias=inp["bias"], softplus=True, dt_min=lo, dt_max=hi)
    y_ref, S_ref = oracle.step(inp["x"], dtp, inp["A"], inp["B"], inp["C"], inp["D"], inp["S"])
    tol = TOL["fp32"] if dtype == torch.float32 else TOL["bf16"]
    assert rel_err(y, y_ref) <= tol
    assert rel_err(S, S_ref) <= TOL["fp32"]


def test_step_without_transform_uses_dt_as_given():
    # dt = 0 freezes the state and leaves y = S C + D x
    inp = _step_inputs(9, 2, 4, 16, 32, 1, torch.float32)
    inp["dt"] = torch.zeros_like(inp["dt"])
    y, S = _run_step(inp)
    np.testing.assert_array_equal(S, inp["S"].numpy())
    y_ref, _ = oracle.step(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["S"])
    assert rel_err(y, y_ref) <= TOL["fp32"]


# ---------------------------------------------------------------- scan + transform

SCAN_CASES = [
    # (workload, algo, overrides)
    (0, "simt", dict(seed=5, batch=1, seqlen=256, nheads=2)),
    (1, "tc", dict(seed=6, batch=2, seqlen=700, nheads=6, init_states=True)),
    (1, "tc2", dict(seed=7, batch=2, seqlen=700, nheads=6, init_states=True)),
    (1, "simt", dict(seed=8, batch=1, seqlen=300, nheads=4)),
    (4, "tc", dict(seed=9, seqlen=1000, nheads=8, init_states=True,
                   segment_lengths=[300, 1, 450, 0, 249])),
    (4, "simt", dict(seed=10, seqlen=600, nheads=4, segment_lengths=[100, 380, 120])),
    (3, "tc2", dict(seed=11, batch=1, seqlen=512, nheads=8)),
    # few long lanes: split between CTAs (state-only pre run, fold, main run)
    (1, "tc", dict(seed=13, batch=1, seqlen=4096, nheads=8, init_states=True)),
    (3, "tc", dict(seed=14, batch=1, seqlen=4096, nheads=8, init_states=True)),
]


@pytest.mark.parametrize("case", SCAN_CASES, ids=lambda c: f"w{c[0]}-{c[1]}-L{c[2]['seqlen']}")
@pytest.mark.parametrize("limit", [None, (0.003, 0.06)])
def test_scan_with_dt_transform(case, limit):
    import mamba_ssd_layer_03_b300 as ssd
    wi, algo, kw = case
    inp = ssd_synth.make_inputs(ssd_synth.WORKLOADS[wi], **kw)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    shape = ssd.make_shape(inp["batch"], inp["seqlen"], inp["nheads"], inp["headdim"],
                           inp["dstate"], inp["ngroups"], inp["chunk"], inp["nseq"],
                           inp["x"].dtype, algo)
    if ssd.load_library().ssd_resolve_algo(shape) < 0:
        pytest.skip(f"{algo} does not take this shape")
    y, fin = ssd.ssd_scan(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], d["D"], inp["chunk"],
                          d["initial_states"], d["cu_seqlens"], True, algo, check_status=True,
                          dt_bias=d["dt_bias"], dt_softplus=True, dt_limit=limit)
    torch.cuda.synchronize()
    lo, hi = (0.0, np.inf) if limit is None else limit
    dtp = oracle.dt_transform(inp["dt_raw"], bias=inp["dt_bias"], softplus=True, dt_min=lo,
                              dt_max=hi)
    tol = TOL[inp["dtype"]]
    y_ref, fin_ref = oracle.recurrent(inp["x"], dtp, inp["A"], inp["B"], inp["C"], inp["D"],
                                      inp["initial_states"], inp["cu_seqlens"])
    assert rel_err(y.float().cpu().numpy(), y_ref) <= tol
    assert rel_err(fin.cpu().numpy(), fin_ref) <= tol
    # without D: the scan term alone, which D x would otherwise dominate
    y0, _ = ssd.ssd_scan(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], None, inp["chunk"],
                         d["initial_states"], d["cu_seqlens"], False, algo, check_status=True,
                         dt_bias=d["dt_bias"], dt_softplus=True, dt_limit=limit)
    torch.cuda.synchronize()
    y0_ref, _ = oracle.recurrent(inp["x"], dtp, inp["A"], inp["B"], inp["C"], None,
                                 inp["initial_states"], inp["cu_seqlens"])
    assert rel_err(y0.float().cpu().numpy(), y0_ref) <= tol


def test_scan_transform_equals_pretransformed_dt():
    """With softplus and the generator's bias, the transform reproduces the
    generator's own dt, so the two calls agree to the dt rounding."""
    import mamba_ssd_layer_03_b300 as ssd
    inp = ssd_synth.make_inputs(ssd_synth.WORKLOADS[1], seed=12, batch=2, seqlen=512, nheads=6)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y1, f1 = ssd.ssd_scan(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], 256, algo="tc",
                          check_status=True)
    y2, f2 = ssd.ssd_scan(d["x"], d["dt_raw"], d["A"], d["B"], d["C"], d["D"], 256, algo="tc",
                          check_status=True, dt_bias=d["dt_bias"], dt_softplus=True)
    torch.cuda.synchronize()
    assert rel_err(y2.float().cpu().numpy(), y1.float().cpu().numpy()) <= 1e-2
    assert rel_err(f2.cpu().numpy(), f1.cpu().numpy()) <= 1e-4
