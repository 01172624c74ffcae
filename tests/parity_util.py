"""Helpers shared by the GPU parity tests: run the CUDA path, run the oracle on
the same inputs (whole problem or sampled (sequence, head) units), compare."""
import numpy as np
import torch

import oracle

TOL = {"fp32": 1e-5, "bf16": 2e-2}


def rel_err(got, ref) -> float:
    """max |got - ref| / max |ref| (the tolerance measure of the SSD scan)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    den = np.abs(ref).max()
    num = np.abs(got - ref).max()
    if den == 0:
        return float(num)
    return float(num / den)


def to_device(inp, dev="cuda"):
    out = dict(inp)
    for k in ("x", "dt", "A", "B", "C", "D", "initial_states", "cu_seqlens"):
        if out.get(k) is not None:
            out[k] = out[k].to(dev)
    return out


def run_gpu(inp, chunk=None, algo="auto", D=True, init=True, final=True):
    import mamba_ssd_layer_03_b300 as ssd
    d = to_device(inp)
    y, fin = ssd.ssd_scan(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"] if D else None,
                          chunk or inp["chunk"], d["initial_states"] if init else None,
                          d["cu_seqlens"], return_final_states=final, algo=algo,
                          check_status=True)
    torch.cuda.synchronize()
    return (y.float().cpu().numpy(),
            None if fin is None else fin.cpu().numpy())


def oracle_full(inp, D=True, init=True):
    return oracle.recurrent(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                            inp["D"] if D else None,
                            inp["initial_states"] if init else None, inp["cu_seqlens"])


def unit_slices(inp, s, h):
    """Index ranges of (sequence s, head h): (row, t0, t1, group)."""
    H, G = inp["nheads"], inp["ngroups"]
    g = h // (H // G)
    if inp["cu_seqlens"] is not None:
        cu = inp["cu_seqlens"]
        return 0, int(cu[s]), int(cu[s + 1]), g
    return s, 0, inp["seqlen"], g


def oracle_unit(inp, s, h, D=True, init=True):
    """Oracle result of one (sequence, head) unit from sliced inputs."""
    return oracle.recurrent_unit(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                                 inp["D"] if D else None,
                                 inp["initial_states"] if init else None,
                                 inp["cu_seqlens"], s, h)


def sample_units(inp, n, seed=0):
    rng = np.random.default_rng(seed)
    nseq, H = inp["nseq"], inp["nheads"]
    units = {(0, 0), (nseq - 1, H - 1)}
    while len(units) < min(n, nseq * H):
        units.add((int(rng.integers(nseq)), int(rng.integers(H))))
    return sorted(units)
