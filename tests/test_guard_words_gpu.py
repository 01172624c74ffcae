"""Guard words around the outputs: the kernels write y and final_states exactly
within their documented extents.

compute-sanitizer is not available here, so out-of-bounds writes are looked for
the plain way.  Each output is a view into a larger buffer, and the words
before and after the view hold a fixed bit pattern.  After the scan, the
pattern must be intact and the outputs must match the oracle.  The cases cover
the places where a store could overrun: ragged last blocks (TMA stores and
direct row stores), packed sequences with empty and one-token sequences, lanes
handed between CTAs or split between them, wide lanes, and the two-pass and
SIMT paths.
"""
import numpy as np
import pytest
import torch

import ssd_synth
from parity_util import TOL, oracle_full, rel_err, to_device

pytestmark = pytest.mark.gpu

W = ssd_synth.WORKLOADS
GUARD = 256   # elements on each side (a multiple of 16 bytes for every dtype here)


def guarded(shape, dtype, device):
    """(buffer, view): `view` has `shape` and sits GUARD elements into a
    buffer filled with a fixed pattern (all bits 0x5A)."""
    n = int(np.prod(shape))
    esz = torch.empty((), dtype=dtype).element_size()
    raw = torch.full(((n + 2 * GUARD) * esz,), 0x5A, dtype=torch.uint8, device=device)
    buf = raw.view(dtype)
    return raw, buf[GUARD:GUARD + n].view(shape)


def guards_intact(raw, n, esz) -> bool:
    lo = raw[:GUARD * esz]
    hi = raw[(GUARD + n) * esz:]
    return bool((lo == 0x5A).all().item()) and bool((hi == 0x5A).all().item())


def run_guarded(inp, algo, scan=None):
    """The scan into guarded outputs; returns (y, final, y_ok, final_ok)."""
    import mamba_ssd_layer_03_b300 as ssd
    scan = scan or ssd.ssd_scan
    dev = "cuda" if scan is ssd.ssd_scan else "cpu"
    d = to_device(inp, dev)
    x = d["x"]
    b, L, H, P = x.shape
    N = d["B"].shape[3]
    nseq = inp["nseq"]
    y_raw, y = guarded((b, L, H, P), x.dtype, dev)
    f_raw, fin = guarded((nseq, H, P, N), torch.float32, dev)
    scan(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], inp["chunk"], d["initial_states"],
         d["cu_seqlens"], True, algo, out=y, final_out=fin, check_status=True)
    if dev == "cuda":
        torch.cuda.synchronize()
    y_ok = guards_intact(y_raw, y.numel(), y.element_size())
    f_ok = guards_intact(f_raw, fin.numel(), 4)
    return y.float().cpu().numpy(), fin.cpu().numpy(), y_ok, f_ok


CASES = [
    # (workload, algo, overrides)
    (1, "tc", dict(seed=71, batch=2, seqlen=700, nheads=6, init_states=True)),      # ragged last block
    (1, "tc", dict(seed=72, batch=1, seqlen=4096, nheads=8, init_states=True)),     # split lanes
    (1, "tc", dict(seed=73, batch=3, seqlen=1000, nheads=120, init_states=True)),   # more lanes than SMs
    (3, "tc", dict(seed=74, batch=1, seqlen=300, nheads=8, init_states=True)),      # wide lanes, ragged
    (4, "tc", dict(seed=75, seqlen=1000, nheads=4, init_states=True,
                   segment_lengths=[300, 1, 450, 0, 249])),                         # packed sequences
    (1, "tc2", dict(seed=76, batch=2, seqlen=700, nheads=6, init_states=True)),
    (0, "simt", dict(seed=77, batch=2, seqlen=200, nheads=2)),
    (4, "simt", dict(seed=78, seqlen=600, nheads=2, segment_lengths=[100, 0, 380, 120])),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"w{c[0]}-{c[1]}-L{c[2]['seqlen']}")
def test_outputs_stay_inside_their_extents(case):
    import mamba_ssd_layer_03_b300 as ssd
    wi, algo, kw = case
    inp = ssd_synth.make_inputs(W[wi], **kw)
    shape = ssd.make_shape(inp["batch"], inp["seqlen"], inp["nheads"], inp["headdim"], inp["dstate"],
                           inp["ngroups"], inp["chunk"], inp["nseq"], inp["x"].dtype, algo)
    if ssd.load_library().ssd_resolve_algo(shape) < 0:
        pytest.skip(f"{algo} does not take this shape")
    y, fin, y_ok, f_ok = run_guarded(inp, algo)
    assert y_ok, "a kernel wrote outside y"
    assert f_ok, "a kernel wrote outside final_states"
    y_ref, f_ref = oracle_full(inp)
    tol = TOL[inp["dtype"]]
    assert rel_err(y, y_ref) <= tol
    assert rel_err(fin, f_ref) <= tol
