"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on
identical seeded inputs.  Bar: max-abs error / max-abs oracle value <= 1e-5
for fp32 inputs and <= 2e-2 for bf16 inputs, on y and on final_states."""
import numpy as np
import pytest
import torch

import ssd_synth
from parity_util import (TOL, oracle_full, oracle_unit, rel_err, run_gpu, sample_units,
                         unit_slices)

pytestmark = pytest.mark.gpu

W = ssd_synth.WORKLOADS
ALGOS = ["simt", "tc", "tc2"]


def _algo_ok(inp, algo, chunk=None):
    """Whether `algo` takes this input: "tc" is the fused tensor-core kernel
    (bf16, headdim 64, dstate 128, any chunk size, packed sequences too) or,
    for other tensor-core shapes, the two-pass kernels; "tc2" is the two-pass
    kernels (bf16, headdim 64, dstate 128/256, chunk 128/256, no packing)."""
    if algo == "simt":
        return True
    import mamba_ssd_layer_03_b300 as ssd
    dt = torch.float32 if inp["dtype"] == "fp32" else torch.bfloat16
    shape = ssd.make_shape(inp["batch"], inp["seqlen"], inp["nheads"], inp["headdim"],
                           inp["dstate"], inp["ngroups"], chunk or inp["chunk"], inp["nseq"], dt,
                           algo)
    try:
        resolved = ssd.resolve_algo(shape)
    except ssd.SsdError as e:
        if e.code == 2:
            return False
        raise
    return resolved == "tc" or inp["cu_seqlens"] is None


def _compare_full(inp, algo, chunk=None, D=True, init=True):
    if not _algo_ok(inp, algo, chunk):
        pytest.skip(f"{algo} path does not take this input")
    tol = TOL[inp["dtype"]]
    y, fin = run_gpu(inp, chunk=chunk, algo=algo, D=D, init=init)
    y_ref, fin_ref = oracle_full(inp, D=D, init=init)
    ey, ef = rel_err(y, y_ref), rel_err(fin, fin_ref)
    assert ey <= tol, f"y rel err {ey:.3e} > {tol}"
    assert ef <= tol, f"final_states rel err {ef:.3e} > {tol}"
    if D:
        # D x is most of |y| at these scales (B, C ~ N(0, 1/N), dt ~ 1e-3..1e-1),
        # so the bar is checked once more on the scan term alone.
        y0, _ = run_gpu(inp, chunk=chunk, algo=algo, D=False, init=init, final=False)
        y0_ref, _ = oracle_full(inp, D=False, init=init)
        e0 = rel_err(y0, y0_ref)
        assert e0 <= tol, f"y (D = 0) rel err {e0:.3e} > {tol}"
    return ey, ef


@pytest.mark.parametrize("algo", ALGOS)
def test_tiny_fp32_workload_full(algo):
    inp = ssd_synth.make_inputs(W[0], seed=0)
    if not _algo_ok(inp, algo):
        pytest.skip("tensor-core path is bf16 only")
    _compare_full(inp, algo)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("chunk", [64, 128, 256])
def test_chunk_size_independence_fp32(algo, chunk):
    inp = ssd_synth.make_inputs(W[0], seed=1, seqlen=300, init_states=True)
    if not _algo_ok(inp, algo):
        pytest.skip("tensor-core path is bf16 only")
    _compare_full(inp, algo, chunk=chunk)


# Reduced-length versions of the bf16 workloads: several chunks plus a ragged
# tail, small enough for the whole oracle.
REDUCED = [
    (1, dict(batch=2, seqlen=1000, nheads=6)),
    (2, dict(batch=2, seqlen=777, nheads=5)),
    (3, dict(batch=2, seqlen=1100, nheads=8)),
    (4, dict(batch=1, seqlen=2000, nheads=4, segment_lengths=[1, 255, 256, 300, 64, 1, 1123])),
]


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("wi,kw", REDUCED, ids=[f"w{w}" for w, _ in REDUCED])
def test_reduced_workloads_full(algo, wi, kw):
    inp = ssd_synth.make_inputs(W[wi], seed=wi, **kw)
    _compare_full(inp, algo)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("chunk", [64, 128, 256])
def test_chunk_size_independence_bf16(algo, chunk):
    inp = ssd_synth.make_inputs(W[3], seed=5, batch=1, seqlen=700, nheads=8)
    _compare_full(inp, algo, chunk=chunk)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("L", [1, 63, 64, 65, 256, 257])
def test_short_and_boundary_lengths(algo, L):
    inp = ssd_synth.make_inputs(W[1], seed=L, batch=2, seqlen=L, nheads=3, init_states=True)
    _compare_full(inp, algo, chunk=64)


@pytest.mark.parametrize("chunk", [128, 256])
@pytest.mark.parametrize("L", [1, 2, 127, 128, 129, 255, 256, 257, 513, 1023])
def test_short_and_boundary_lengths_tc_chunks(chunk, L):
    """Lengths around the tensor-core path's 128-token blocks and chunk ends,
    at the chunk sizes it takes (both paths run)."""
    inp = ssd_synth.make_inputs(W[1], seed=1000 + L, batch=2, seqlen=L, nheads=4, init_states=True)
    for algo in ALGOS:
        _compare_full(inp, algo, chunk=chunk)


@pytest.mark.parametrize("segs", [None, [130, 1, 600, 257, 512, 12]])
def test_lanes_split_between_ctas(segs):
    """More (sequence, head pair) lanes than SMs, so that the fused kernel
    hands the running state of a lane from one CTA to the next."""
    if segs is None:
        inp = ssd_synth.make_inputs(W[1], seed=31, batch=2, seqlen=300, nheads=160,
                                    init_states=True)
    else:
        inp = ssd_synth.make_inputs(W[4], seed=32, seqlen=sum(segs), nheads=64,
                                    init_states=True, segment_lengths=segs)
    _compare_full(inp, "tc")


@pytest.mark.parametrize("algo", ALGOS)
def test_optional_arguments_absent(algo):
    inp = ssd_synth.make_inputs(W[1], seed=9, batch=1, seqlen=513, nheads=4, init_states=True)
    if not _algo_ok(inp, algo):
        pytest.skip(f"{algo} path does not take this input")
    y, fin = run_gpu(inp, algo=algo, D=False, init=False, final=False)
    assert fin is None
    y_ref, _ = oracle_full(inp, D=False, init=False)
    assert rel_err(y, y_ref) <= TOL["bf16"]


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("segs", [
    [64, 64, 64, 64],            # boundaries exactly on chunk ends
    [1] * 70,                    # many single-token sequences
    [100, 0, 0, 156, 0],         # empty sequences
    [1000],                      # one sequence across many chunks
    [5, 250, 7, 500, 2, 260],    # mixed
])
def test_varlen_edges_with_initial_states(algo, segs):
    L = sum(segs)
    inp = ssd_synth.make_inputs(W[4], seed=len(segs), seqlen=L, nheads=3,
                                init_states=True, segment_lengths=segs)
    _compare_full(inp, algo, chunk=64)


@pytest.mark.parametrize("algo", ALGOS)
def test_varlen_packed_equals_separate_runs(algo):
    segs = [300, 17, 451]
    inp = ssd_synth.make_inputs(W[4], seed=77, seqlen=sum(segs), nheads=4,
                                init_states=True, segment_lengths=segs)
    if not _algo_ok(inp, algo):
        pytest.skip(f"{algo} path does not take this input")
    y, fin = run_gpu(inp, algo=algo)
    cu = inp["cu_seqlens"]
    for s in range(len(segs)):
        a, b = int(cu[s]), int(cu[s + 1])
        sep = dict(inp)
        for k in ("x", "dt", "B", "C"):
            sep[k] = inp[k][:, a:b].contiguous()
        sep["cu_seqlens"] = None
        sep["initial_states"] = inp["initial_states"][s:s + 1].contiguous()
        sep["seqlen"], sep["nseq"] = b - a, 1
        ys, fs = run_gpu(sep, algo=algo)
        assert rel_err(y[:, a:b], ys) <= 1e-2
        assert rel_err(fin[s:s + 1], fs) <= 1e-2


@pytest.mark.parametrize("algo", ALGOS)
def test_split_invariance_through_states(algo):
    inp = ssd_synth.make_inputs(W[3], seed=11, batch=2, seqlen=900, nheads=8)
    if not _algo_ok(inp, algo):
        pytest.skip(f"{algo} path does not take this input")
    y, fin = run_gpu(inp, algo=algo)
    t0 = 384
    first, second = dict(inp), dict(inp)
    for k in ("x", "dt", "B", "C"):
        first[k] = inp[k][:, :t0].contiguous()
        second[k] = inp[k][:, t0:].contiguous()
    first["seqlen"], second["seqlen"] = t0, 900 - t0
    y1, f1 = run_gpu(first, algo=algo)
    second["initial_states"] = torch.from_numpy(f1)
    y2, f2 = run_gpu(second, algo=algo)
    assert rel_err(np.concatenate([y1, y2], axis=1), y) <= 1e-2
    assert rel_err(f2, fin) <= 1e-2


@pytest.mark.parametrize("algo", ALGOS)
def test_dt_zero_freezes_state(algo):
    inp = ssd_synth.make_inputs(W[1], seed=3, batch=1, seqlen=300, nheads=2, init_states=True)
    inp["dt"] = torch.zeros_like(inp["dt"])
    if not _algo_ok(inp, algo):
        pytest.skip(f"{algo} path does not take this input")
    y, fin = run_gpu(inp, algo=algo)
    assert np.array_equal(fin, inp["initial_states"].numpy())
    _compare_full(inp, algo)


# ---- full-size workloads, in the launch configuration the benchmark times ----

@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("wi", [1, 2, 3, 4])
def test_full_size_workload_sampled(algo, wi):
    inp = ssd_synth.make_inputs(W[wi], seed=0)
    if not _algo_ok(inp, algo):
        pytest.skip(f"{algo} path does not take this input")
    tol = TOL[inp["dtype"]]
    y, fin = run_gpu(inp, algo=algo)
    y0, _ = run_gpu(inp, algo=algo, D=False, final=False)
    assert np.isfinite(y).all() and np.isfinite(y0).all()
    for (s, h) in sample_units(inp, 6, seed=wi):
        yu, fu = oracle_unit(inp, s, h)
        y0u, _ = oracle_unit(inp, s, h, D=False)
        row, t0, t1, _ = unit_slices(inp, s, h)
        assert rel_err(y[row, t0:t1, h], yu) <= tol, (s, h)
        assert rel_err(y0[row, t0:t1, h], y0u) <= tol, (s, h, "D = 0")
        assert rel_err(fin[s, h], fu) <= tol, (s, h)


@pytest.mark.parametrize("algo", ALGOS)
def test_full_size_workload1_complete(algo):
    inp = ssd_synth.make_inputs(W[1], seed=0)
    _compare_full(inp, algo)


def test_malformed_cu_seqlens_reports_status():
    import mamba_ssd_layer_03_b300 as ssd
    inp = ssd_synth.make_inputs(W[4], seed=1, seqlen=300, nheads=2, segment_lengths=[100, 200])
    bad = torch.tensor([0, 200, 100, 300], dtype=torch.int32)  # decreasing
    dev = "cuda"
    S0 = torch.zeros(3, 2, 64, 128, device=dev)
    with pytest.raises(ssd.SsdError) as ei:
        ssd.ssd_scan(inp["x"].to(dev), inp["dt"].to(dev), inp["A"].to(dev), inp["B"].to(dev),
                     inp["C"].to(dev), None, 64, S0, bad.to(dev), check_status=True)
    assert ei.value.code == 6
    # the context is still usable
    y, _ = run_gpu(inp)
    assert np.isfinite(y).all()


def test_empty_inputs():
    import mamba_ssd_layer_03_b300 as ssd
    dev = "cuda"
    for b, L in [(2, 0), (0, 16)]:
        x = torch.zeros(b, L, 2, 64, dtype=torch.bfloat16, device=dev)
        dt = torch.zeros(b, L, 2, device=dev)
        A = -torch.ones(2, device=dev)
        B = torch.zeros(b, L, 1, 128, dtype=torch.bfloat16, device=dev)
        S0 = torch.randn(b, 2, 64, 128, device=dev)
        y, fin = ssd.ssd_scan(x, dt, A, B, B.clone(), None, 256, S0 if b else None,
                              check_status=True)
        assert y.shape == x.shape
        if b:
            assert torch.equal(fin, S0)


def test_host_buffers_round_trip():
    import mamba_ssd_layer_03_b300 as ssd
    inp = ssd_synth.make_inputs(W[1], seed=4, batch=1, seqlen=600, nheads=3)
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y, fin = ssd.ssd_scan(pin["x"], pin["dt"], pin["A"], pin["B"], pin["C"], pin["D"], 256)
    assert y.device.type == "cpu" and fin.device.type == "cpu"
    y_ref, f_ref = oracle_full(inp)
    assert rel_err(y.float().numpy(), y_ref) <= TOL["bf16"]
    assert rel_err(fin.numpy(), f_ref) <= TOL["bf16"]


# ---------------------------------------------------------------- wide lanes
# dstate 256: the fused kernel runs one head per lane, the state's two
# 128-row halves in the two warpgroups.

@pytest.mark.parametrize("kw", [
    dict(seed=41, batch=4, seqlen=400, nheads=64, init_states=True),    # 256 lanes > SMs: handoffs
    dict(seed=42, batch=1, seqlen=130, nheads=8, init_states=False),    # one block and a 2-token tail
])
def test_wide_lanes_fused(kw):
    inp = ssd_synth.make_inputs(W[3], **kw)
    _compare_full(inp, "tc")


@pytest.mark.parametrize("segs", [[300, 1, 0, 450, 249], [128] * 6])
def test_wide_lanes_packed_sequences(segs):
    inp = ssd_synth.make_inputs(W[3], seed=43, batch=1, seqlen=sum(segs), nheads=16,
                                init_states=True, segment_lengths=segs)
    _compare_full(inp, "tc")


# ---------------------------------------------------------------- split lanes
# Fewer lanes than SMs with long sequences: the fused kernel splits every lane
# between several CTAs.  A state-only first run records each CTA's partial
# state and decay; the records are folded into each split's start state; the
# second run produces y.

@pytest.mark.parametrize("wi,kw", [
    (1, dict(seed=61, batch=1, seqlen=8192, nheads=24, init_states=True)),   # 12 lanes on all SMs, ranges straddle
    (1, dict(seed=62, batch=1, seqlen=6000, nheads=6, init_states=True)),    # 3 lanes, ragged tail
    (3, dict(seed=63, batch=1, seqlen=8192, nheads=8, init_states=True)),    # wide lanes
    (1, dict(seed=64, batch=2, seqlen=2048, nheads=24, init_states=True)),   # 4 blocks per CTA, lane-aligned
    # wide lanes, several heads per B/C group (8 groups): CTAs in sets of 4, 3
    # and 6 take the same range of a group's lanes, one lane each
    (3, dict(seed=65, batch=1, seqlen=4096, nheads=32, init_states=True)),
    (3, dict(seed=66, batch=2, seqlen=2500, nheads=24, init_states=True)),
    (3, dict(seed=67, batch=1, seqlen=3000, nheads=48, init_states=False)),
], ids=["narrow", "straddle", "wide", "four_blocks", "wide_sets4", "wide_sets3_ragged", "wide_sets6"])
def test_split_lanes_two_runs(wi, kw):
    inp = ssd_synth.make_inputs(W[wi], **kw)
    _compare_full(inp, "tc")


# ---------------------------------------------------------------- strong decay
# Heads whose decay over a few tokens is enormous.  With A = -16 and a constant
# step dt, 32 tokens decay by exp(-512 dt): about e^-51 at dt = 0.1, e^-77 at
# dt = 0.15 and e^-512 at dt = 1.  The fused kernel factors the masked block
# at 32-token sub-blocks and changes method once a sub-block's decay is too
# large for the factored form, so these cases run both of its methods and the
# boundary between them; "mixed" gives the two heads of a lane different
# regimes.  The last case is the limit Delta -> infinity, which replaces the
# state by the current input (Mamba-1 walkthrough "Mamba: Linear-Time
# Sequence Modeling with Selective State Spaces", sections 三 2.3 "边界重置"
# and 三 3).

def _strong_decay(inp, regime, seed):
    H = inp["nheads"]
    g = torch.Generator().manual_seed(seed)
    shape = inp["dt"].shape
    if regime == "mixed":
        # per head: 0.02 (weak), 0.1, 0.15, 1.0, cycling, plus noise
        base = torch.tensor([0.02, 0.1, 0.15, 1.0])[torch.arange(H) % 4]
        dt = base * (1.0 + 0.2 * torch.rand(shape, generator=g))
    else:
        dt = torch.full(shape, float(regime))
    inp = dict(inp)
    inp["dt"] = dt.contiguous()
    inp["A"] = torch.full((H,), -16.0)
    return inp


STRONG = [
    (1, dict(batch=2, seqlen=700, nheads=6, init_states=True)),     # narrow lanes, one run
    (3, dict(batch=1, seqlen=520, nheads=8, init_states=True)),     # wide lanes (dstate 256)
    (1, dict(batch=1, seqlen=4096, nheads=8, init_states=True)),    # narrow, split lanes
    (3, dict(batch=1, seqlen=4096, nheads=8, init_states=True)),    # wide, split lanes
]


@pytest.mark.parametrize("regime", ["0.1", "0.15", "1.0", "mixed"])
@pytest.mark.parametrize("wi,kw", STRONG, ids=["narrow", "wide", "narrow_split", "wide_split"])
def test_strong_decay_fused(wi, kw, regime):
    inp = _strong_decay(ssd_synth.make_inputs(W[wi], seed=90 + wi, **kw), regime, seed=wi)
    _compare_full(inp, "tc")


@pytest.mark.parametrize("algo", ["simt", "tc2"])
@pytest.mark.parametrize("regime", ["0.15", "mixed"])
def test_strong_decay_other_paths(algo, regime):
    inp = _strong_decay(ssd_synth.make_inputs(W[1], seed=95, batch=2, seqlen=600, nheads=4,
                                              init_states=True), regime, seed=7)
    _compare_full(inp, algo)


@pytest.mark.parametrize("wi", [1, 3])
@pytest.mark.parametrize("algo", ALGOS)
def test_huge_dt_replaces_state(algo, wi):
    """dt = 50 with A = -1: every token's decay is e^-50, so after each token
    the state is dt x_t (outer) B_t to well within the tolerance, and y_t is
    C_t . (dt x_t (outer) B_t) + D x_t."""
    inp = ssd_synth.make_inputs(W[wi], seed=97, batch=1, seqlen=333, nheads=8, init_states=True)
    inp["dt"] = torch.full_like(inp["dt"], 50.0)
    inp["A"] = torch.full((inp["nheads"],), -1.0)
    ey, ef = _compare_full(inp, algo)
    y, fin = run_gpu(inp, algo=algo)
    H, G = inp["nheads"], inp["ngroups"]
    x = inp["x"].double().numpy()
    Bm, Cm = inp["B"].double().numpy(), inp["C"].double().numpy()
    D = inp["D"].double().numpy()
    for h in range(H):
        g = h // (H // G)
        S_last = 50.0 * np.outer(x[0, -1, h], Bm[0, -1, g])
        assert rel_err(fin[0, h], S_last) <= TOL["bf16"], h
        y_exp = 50.0 * x[0, :, h] * (Bm[0, :, g] * Cm[0, :, g]).sum(-1)[:, None] + D[h] * x[0, :, h]
        assert rel_err(y[0, :, h], y_exp) <= TOL["bf16"], h
