"""Pins for the CPU oracle: checks against things other than the oracle itself.

* hand-derived golden fixtures (tests/golden/*.json);
* closed forms: A = 0 gives prefix sums, constant decay gives a geometric
  series, dt = 0 freezes the state, L = 1;
* the duality of the recurrent and semiseparable-matrix forms (two separately
  written formulations of the same map);
* invariants: splitting a sequence and passing final_states as initial_states
  reproduces the unsplit run; packed sequences equal separate runs; linearity
  in (x, initial_states); the unit subset equals the full run;
* a one-sided check that a huge dt with A < 0 replaces the state by the
  current input (boundary resetting, Mamba-1 walkthrough section 三 2.3);
* planted mistakes in the oracle are caught by at least one of these pins;
* the block decomposition (chunked form) agrees with both formulations at
  every chunk size, its steps meet their closed forms, and a mistake planted
  in any one step breaks that agreement.
"""
import glob
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import ssd_synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(seed, b=1, L=40, H=4, P=3, N=5, G=2, init=True, D=True, cu=None):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(b, L, H, P, generator=g, dtype=torch.float64)
    dt = torch.rand(b, L, H, generator=g, dtype=torch.float64) * 0.5 + 0.01
    A = -torch.rand(H, generator=g, dtype=torch.float64) * 3 - 0.1
    B = torch.randn(b, L, G, N, generator=g, dtype=torch.float64)
    C = torch.randn(b, L, G, N, generator=g, dtype=torch.float64)
    Dv = torch.randn(H, generator=g, dtype=torch.float64) if D else None
    nseq = (len(cu) - 1) if cu is not None else b
    S0 = torch.randn(nseq, H, P, N, generator=g, dtype=torch.float64) if init else None
    cuv = None if cu is None else torch.tensor(cu, dtype=torch.int32)
    return dict(x=x, dt=dt, A=A, B=B, C=C, D=Dv, initial_states=S0, cu_seqlens=cuv)


def _golden_cases():
    return sorted(glob.glob(os.path.join(GOLDEN, "*.json")))


FORMS = {
    "recurrent": oracle.recurrent,
    "quadratic": oracle.quadratic,
    "chunked1": lambda **kw: oracle.chunked(chunk=1, **kw),
    "chunked2": lambda **kw: oracle.chunked(chunk=2, **kw),
    "chunked64": lambda **kw: oracle.chunked(chunk=64, **kw),
}


@pytest.mark.parametrize("path", _golden_cases(), ids=lambda p: os.path.basename(p))
@pytest.mark.parametrize("form", sorted(FORMS))
def test_golden_fixture(path, form):
    with open(path) as f:
        g = json.load(f)
    A = np.array(g["A_log2_multiple"]) * math.log(2.0)
    args = dict(x=np.array(g["x"]), dt=np.array(g["dt"]), A=A, B=np.array(g["B"]),
                C=np.array(g["C"]), D=np.array(g["D"]),
                initial_states=None if g["initial_states"] is None else np.array(g["initial_states"]),
                cu_seqlens=g["cu_seqlens"])
    y, fin = FORMS[form](**args)
    np.testing.assert_allclose(y, np.array(g["y"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(fin, np.array(g["final_states"]), rtol=0, atol=1e-12)


def test_prefix_sum_when_A_zero():
    # A = 0, N = P = 1, B = C = dt = 1, D = 0: the state is the running sum of x.
    L = 200
    x = np.random.default_rng(1).standard_normal((1, L, 1, 1))
    ones = np.ones((1, L, 1, 1))
    y, fin = oracle.recurrent(x, np.ones((1, L, 1)), np.zeros(1), ones, ones)
    np.testing.assert_allclose(y[0, :, 0, 0], np.cumsum(x[0, :, 0, 0]), rtol=1e-13, atol=1e-12)
    assert abs(fin[0, 0, 0, 0] - x.sum()) < 1e-11


@pytest.mark.parametrize("dtv,Av", [(0.3, -0.7), (0.05, -4.0), (1.0, -1e-3)])
def test_geometric_closed_form(dtv, Av):
    # Constant a = dt A, N = P = 1, B = C = 1, constant x:
    # y_t = dt x (1 - e^{a (t+1)}) / (1 - e^{a}).
    L, xv = 300, 1.7
    a = dtv * Av
    t = np.arange(L)
    expect = dtv * xv * (1 - np.exp(a * (t + 1))) / (1 - np.exp(a))
    y, _ = oracle.recurrent(np.full((1, L, 1, 1), xv), np.full((1, L, 1), dtv), np.array([Av]),
                            np.ones((1, L, 1, 1)), np.ones((1, L, 1, 1)))
    np.testing.assert_allclose(y[0, :, 0, 0], expect, rtol=1e-12)


def test_dt_zero_freezes_state():
    c = _rand_case(3)
    c["dt"] = torch.zeros_like(c["dt"])
    y, fin = oracle.recurrent(**c)
    S0 = c["initial_states"].numpy()
    C, x, D = c["C"].numpy(), c["x"].numpy(), c["D"].numpy()
    H, G = x.shape[2], C.shape[2]
    for h in range(H):
        g = h // (H // G)
        expect = np.einsum("pn,tn->tp", S0[0, h], C[0, :, g]) + D[h] * x[0, :, h]
        np.testing.assert_allclose(y[0, :, h], expect, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(fin, S0, rtol=0, atol=0)


def test_single_token_closed_form():
    c = _rand_case(4, L=1)
    y, fin = oracle.recurrent(**c)
    x, dt, A, B, C, D, S0 = (c[k].numpy() for k in ("x", "dt", "A", "B", "C", "D", "initial_states"))
    H, G = x.shape[2], B.shape[2]
    for h in range(H):
        g = h // (H // G)
        S = np.exp(dt[0, 0, h] * A[h]) * S0[0, h] + dt[0, 0, h] * np.outer(x[0, 0, h], B[0, 0, g])
        np.testing.assert_allclose(fin[0, h], S, rtol=1e-14, atol=1e-14)
        np.testing.assert_allclose(y[0, 0, h], S @ C[0, 0, g] + D[h] * x[0, 0, h], rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("seed,kw", [
    (10, dict()),
    (11, dict(b=2, G=1, init=False)),
    (12, dict(H=6, G=3, D=False)),
    (13, dict(cu=[0, 7, 8, 25, 40])),
    (14, dict(cu=[0, 1, 40], init=False)),
])
def test_recurrent_equals_quadratic(seed, kw):
    c = _rand_case(seed, **kw)
    y1, f1 = oracle.recurrent(**c)
    y2, f2 = oracle.quadratic(**c)
    np.testing.assert_allclose(y1, y2, rtol=1e-11, atol=1e-11 * np.abs(y2).max())
    np.testing.assert_allclose(f1, f2, rtol=1e-11, atol=1e-11 * np.abs(f2).max())


def test_recurrent_equals_quadratic_tiny_fp32_workload():
    # The whole tiny fp32 workload (L=256, 2 heads, P=N=16) in both forms.
    inp = ssd_synth.make_inputs(ssd_synth.WORKLOADS[0], seed=0)
    args = {k: inp[k] for k in ("x", "dt", "A", "B", "C", "D", "initial_states", "cu_seqlens")}
    y1, f1 = oracle.recurrent(**args)
    y2, f2 = oracle.quadratic(**args)
    assert np.abs(y1 - y2).max() <= 1e-12 * np.abs(y2).max()
    assert np.abs(f1 - f2).max() <= 1e-12 * np.abs(f2).max()


@pytest.mark.parametrize("t0", [1, 17, 39])
def test_split_invariance(t0):
    c = _rand_case(20, b=1)
    y, fin = oracle.recurrent(**c)
    first = {k: (v[:, :t0] if k in ("x", "dt", "B", "C") else v) for k, v in c.items()}
    y1, f1 = oracle.recurrent(**first)
    second = {k: (v[:, t0:] if k in ("x", "dt", "B", "C") else v) for k, v in c.items()}
    second["initial_states"] = f1
    y2, f2 = oracle.recurrent(**second)
    np.testing.assert_allclose(np.concatenate([y1, y2], axis=1), y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(f2, fin, rtol=1e-12, atol=1e-12)


def test_packed_equals_separate():
    cu = [0, 5, 6, 30, 40]
    c = _rand_case(21, cu=cu)
    y, fin = oracle.recurrent(**c)
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        sep = {k: (v[:, a:b] if k in ("x", "dt", "B", "C") else v) for k, v in c.items()}
        sep["cu_seqlens"] = None
        sep["initial_states"] = c["initial_states"][s:s + 1]
        ys, fs = oracle.recurrent(**sep)
        np.testing.assert_allclose(y[:, a:b], ys, rtol=0, atol=0)
        np.testing.assert_allclose(fin[s:s + 1], fs, rtol=0, atol=0)


def test_linearity():
    c1 = _rand_case(30, D=True)
    c2 = _rand_case(31, D=True)
    for k in ("dt", "A", "B", "C", "D"):
        c2[k] = c1[k]
    y1, f1 = oracle.recurrent(**c1)
    y2, f2 = oracle.recurrent(**c2)
    c3 = dict(c1)
    c3["x"] = 2.0 * c1["x"] - 3.0 * c2["x"]
    c3["initial_states"] = 2.0 * c1["initial_states"] - 3.0 * c2["initial_states"]
    y3, f3 = oracle.recurrent(**c3)
    np.testing.assert_allclose(y3, 2 * y1 - 3 * y2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(f3, 2 * f1 - 3 * f2, rtol=1e-12, atol=1e-12)


def test_huge_dt_replaces_state():
    # dt -> infinity with A < 0: exp(dt A) -> 0, so the state after token t is
    # dt_t x_t (outer) B_t regardless of the past (one-sided check).
    c = _rand_case(40, L=10, D=False)
    c["dt"] = torch.full_like(c["dt"], 80.0)
    c["A"] = -torch.ones_like(c["A"])
    y, fin = oracle.recurrent(**c)
    x, B, C = c["x"].numpy(), c["B"].numpy(), c["C"].numpy()
    H, G = x.shape[2], B.shape[2]
    for h in range(H):
        g = h // (H // G)
        S = 80.0 * np.outer(x[0, -1, h], B[0, -1, g])
        np.testing.assert_allclose(fin[0, h], S, rtol=1e-12, atol=1e-12)
        for t in range(10):
            expect = 80.0 * x[0, t, h] * float(B[0, t, g] @ C[0, t, g])
            np.testing.assert_allclose(y[0, t, h], expect, rtol=1e-12, atol=1e-12)


def test_units_subset_matches_full():
    c = _rand_case(50, b=2, H=4, G=2)
    y, fin = oracle.recurrent(**c)
    units = [1, 6]       # (seq 0, head 1) and (seq 1, head 2)
    ys, fs = oracle.recurrent(**c, units=units)
    for u in units:
        s, h = divmod(u, 4)
        np.testing.assert_array_equal(ys[s, :, h], y[s, :, h])
        np.testing.assert_array_equal(fs[s, h], fin[s, h])
    assert np.isnan(ys[0, :, 0]).all()


def test_rejects_bad_cu_seqlens():
    c = _rand_case(60, cu=[0, 10, 40])
    c["cu_seqlens"] = torch.tensor([0, 10, 39], dtype=torch.int32)
    with pytest.raises(ValueError):
        oracle.recurrent(**c)


def _pins_pass(mutation):
    """Run a subset of the pins against a mutated oracle; True if all pass."""
    ok = True
    for path in _golden_cases():
        with open(path) as f:
            g = json.load(f)
        A = np.array(g["A_log2_multiple"]) * math.log(2.0)
        y, fin = oracle.recurrent(np.array(g["x"]), np.array(g["dt"]), A, np.array(g["B"]),
                                  np.array(g["C"]), np.array(g["D"]),
                                  None if g["initial_states"] is None else np.array(g["initial_states"]),
                                  g["cu_seqlens"], mutation=mutation)
        ok &= bool(np.allclose(y, np.array(g["y"]), rtol=0, atol=1e-12))
    c = _rand_case(70, cu=[0, 9, 40])
    y1, _ = oracle.recurrent(**c, mutation=mutation)
    y2, _ = oracle.quadratic(**c)
    ok &= bool(np.allclose(y1, y2, rtol=1e-10, atol=1e-10))
    return ok


@pytest.mark.parametrize("mutation", sorted(oracle.MUTATIONS))
def test_planted_mistakes_are_caught(mutation):
    assert not _pins_pass(mutation), f"mutation {mutation} slipped through the pins"


def test_unmutated_passes_the_same_pins():
    assert _pins_pass(None)


# ---------------------------------------------------------------- step sizes
# The step-size transform Delta = softplus(parameter + s_Delta(x)) (Mamba-1
# walkthrough, section 三(二)), clamp last.  Pinned by values and identities
# of softplus, not by retyping it.

def test_dt_transform_softplus_values():
    z = np.array([[0.0, math.log(math.e - 1.0), 50.0, -50.0]])
    got = oracle.dt_transform(z, softplus=True)
    assert got[0, 0] == pytest.approx(math.log(2.0), rel=1e-15)     # log(1 + 1)
    assert got[0, 1] == pytest.approx(1.0, rel=1e-15)               # log(1 + (e - 1)) = 1
    assert got[0, 2] == pytest.approx(50.0, rel=1e-15)              # log(1 + e^50) = 50 + log1p(e^-50)
    assert got[0, 3] == pytest.approx(math.exp(-50.0), rel=1e-12)   # log(1 + e^-50) ~ e^-50


def test_dt_transform_softplus_identity_and_bias():
    g = torch.Generator().manual_seed(5)
    z = torch.randn(3, 7, 4, generator=g, dtype=torch.float64).numpy() * 6
    sp = oracle.dt_transform(z, softplus=True)
    sm = oracle.dt_transform(-z, softplus=True)
    # softplus(z) - softplus(-z) = z, and softplus(z) > max(z, 0)
    np.testing.assert_allclose(sp - sm, z, rtol=0, atol=1e-12)
    assert np.all(sp > np.maximum(z, 0.0))
    bias = np.array([0.5, -1.0, 2.0, 0.0])
    np.testing.assert_array_equal(oracle.dt_transform(z, bias=bias, softplus=True),
                                  oracle.dt_transform(z + bias, softplus=True))
    # no softplus: the bias alone, then the default clamp at 0 (step sizes are
    # never negative); with no lower bound it is the plain sum
    np.testing.assert_array_equal(oracle.dt_transform(z, bias=bias), np.maximum(z + bias, 0.0))
    np.testing.assert_array_equal(oracle.dt_transform(z, bias=bias, dt_min=-np.inf), z + bias)


def test_dt_transform_clamp():
    z = np.array([[-3.0, 0.2, 0.5, 9.0]])
    np.testing.assert_array_equal(oracle.dt_transform(z, dt_min=0.1, dt_max=1.0),
                                  [[0.1, 0.2, 0.5, 1.0]])
    got = oracle.dt_transform(z, softplus=True, dt_min=0.5, dt_max=2.0)
    assert got[0, 0] == 0.5 and got[0, 3] == 2.0


def test_dt_transform_reproduces_the_generators_step_sizes():
    # the synthetic inputs draw dt = softplus(noise + inv_softplus(dt0)) with
    # torch's softplus; the oracle's transform of (noise, bias) must agree
    w = ssd_synth.WORKLOADS[1]
    raw, bias, dt = ssd_synth.make_dt_parts(w, seed=3, batch=2, seqlen=64, nheads=6)
    got = oracle.dt_transform(raw.double(), bias=bias.double(), softplus=True)
    np.testing.assert_allclose(got, dt.double().numpy(), rtol=1e-6, atol=0)


# ---------------------------------------------------------------- decode step

def test_step_equals_recurrence_token_by_token():
    c = _rand_case(21, b=2, L=9, H=4, P=3, N=5, G=2)
    x, dt, A, B, C, D, S0 = (c[k] for k in ("x", "dt", "A", "B", "C", "D", "initial_states"))
    y_ref, fin_ref = oracle.recurrent(**c)
    S = S0.numpy().copy()
    for t in range(9):
        y, S = oracle.step(x[:, t], dt[:, t], A, B[:, t], C[:, t], D, S)
        np.testing.assert_allclose(y, y_ref[:, t], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S, fin_ref, rtol=1e-12, atol=1e-12)


def test_step_closed_form():
    # one token: S' = e^{dt A} S + dt x B^T, y = S' C + D x, written out by hand
    c = _rand_case(22, b=1, L=1, H=2, P=2, N=3, G=1)
    x, dt, A, B, C, D, S0 = (c[k] for k in ("x", "dt", "A", "B", "C", "D", "initial_states"))
    y, S = oracle.step(x[:, 0], dt[:, 0], A, B[:, 0], C[:, 0], D, S0)
    for h in range(2):
        d = float(dt[0, 0, h])
        Sp = math.exp(d * float(A[h])) * S0[0, h].numpy() + d * np.outer(x[0, 0, h].numpy(), B[0, 0, 0].numpy())
        np.testing.assert_allclose(S[0, h], Sp, rtol=1e-13)
        np.testing.assert_allclose(y[0, h], Sp @ C[0, 0, 0].numpy() + float(D[h]) * x[0, 0, h].numpy(), rtol=1e-13)


# ---------------------------------------------------------------- block decomposition

def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


@pytest.mark.parametrize("chunk", [1, 2, 3, 7, 16, 40, 64])
@pytest.mark.parametrize("seed", [0, 1])
def test_chunked_equals_recurrent(chunk, seed):
    case = _rand_case(seed, b=2, L=40, H=4, P=3, N=5, G=2)
    yr, fr = oracle.recurrent(**case)
    yc, fc = oracle.chunked(chunk=chunk, **case)
    assert _rel(yc, yr) < 1e-12 and _rel(fc, fr) < 1e-12


@pytest.mark.parametrize("chunk", [1, 3, 8])
def test_chunked_equals_quadratic_packed(chunk):
    # packed sequences, one of them empty and one a single token: chunks restart
    # at every sequence start
    case = _rand_case(5, b=1, L=23, H=2, P=2, N=3, G=1, cu=[0, 9, 9, 10, 23])
    yq, fq = oracle.quadratic(**case)
    yc, fc = oracle.chunked(chunk=chunk, **case)
    assert _rel(yc, yq) < 1e-12 and _rel(fc, fq) < 1e-12


def test_chunk_state_closed_forms():
    rng = np.random.default_rng(3)
    X, Bm = rng.standard_normal((1, 4)), rng.standard_normal((1, 6))
    dtv = np.array([0.3])
    # one token: its own contribution dt x (outer) B, undecayed
    S = oracle.chunk_state(Bm, X, dtv, oracle.chunk_decay(dtv * -2.0))
    np.testing.assert_allclose(S, 0.3 * np.outer(X[0], Bm[0]), rtol=1e-15)
    # A = 0: no decay, the plain sum of dt_j x_j (outer) B_j
    X, Bm, dtv = rng.standard_normal((5, 4)), rng.standard_normal((5, 6)), rng.uniform(0.1, 1, 5)
    S = oracle.chunk_state(Bm, X, dtv, oracle.chunk_decay(np.zeros(5)))
    np.testing.assert_allclose(S, sum(dtv[j] * np.outer(X[j], Bm[j]) for j in range(5)), rtol=1e-13)
    # first token of two, decay a_1 = ln(1/2) applied to it once
    X, Bm, dtv = np.ones((2, 1)), np.ones((2, 1)), np.ones(2)
    S = oracle.chunk_state(Bm, X, dtv, oracle.chunk_decay(np.array([math.log(0.25), math.log(0.5)])))
    np.testing.assert_allclose(S, [[0.5 + 1.0]], rtol=1e-15)


def test_state_passing_closed_forms():
    S0 = np.full((2, 2), 3.0)
    zeros = [np.zeros((2, 2))] * 3
    entries, final = oracle.state_passing(zeros, [math.log(0.5)] * 3, S0)
    # no input: the entry states halve from chunk to chunk
    for c, e in enumerate(entries):
        np.testing.assert_allclose(e, S0 * 0.5 ** c, rtol=1e-15)
    np.testing.assert_allclose(final, S0 / 8, rtol=1e-15)
    # no decay: the entry states are prefix sums of the chunk states
    S = [np.full((2, 2), float(c + 1)) for c in range(3)]
    entries, final = oracle.state_passing(S, [0.0] * 3, np.zeros((2, 2)))
    np.testing.assert_allclose(entries[2], np.full((2, 2), 3.0))
    np.testing.assert_allclose(final, np.full((2, 2), 6.0))


def test_chunk_output_closed_forms():
    rng = np.random.default_rng(4)
    Cc, Bc, Xc = rng.standard_normal((1, 5)), rng.standard_normal((1, 5)), rng.standard_normal((1, 3))
    # one token, zero entry state: (C . B) dt x + D x
    y = oracle.chunk_output(Cc, Bc, Xc, np.array([0.2]), np.array([-0.7]), np.zeros((3, 5)), 1.5)
    np.testing.assert_allclose(y, (Cc[0] @ Bc[0]) * 0.2 * Xc + 1.5 * Xc, rtol=1e-14)
    # dt = 0 everywhere: only the entry state, undecayed, read through C
    H = rng.standard_normal((3, 5))
    Cc, Bc, Xc = rng.standard_normal((4, 5)), rng.standard_normal((4, 5)), rng.standard_normal((4, 3))
    y = oracle.chunk_output(Cc, Bc, Xc, np.zeros(4), np.zeros(4), H, None)
    np.testing.assert_allclose(y, Cc @ H.T, rtol=1e-14)


def _planted(monkeypatch, step, fn):
    monkeypatch.setattr(oracle, step, fn)


PLANTED = {
    # the entry state's decay forgotten between chunks
    "no_decay_between_chunks": ("state_passing", lambda S, e, S0: _STATE_PASSING(S, [0.0] * len(e), S0)),
    # the chunk state weighted by the decay from the chunk start instead of to its end
    "state_weight_reversed": ("chunk_state", lambda Bc, Xc, dtc, cs: ((Xc * (np.exp(cs - cs[0]) * dtc)[:, None]).T @ Bc)),
    # the mask's diagonal dropped (j < i instead of j <= i)
    "strict_mask": ("chunk_output", lambda Cc, Bc, Xc, dtc, cs, He, Dh: _CHUNK_OUTPUT(Cc, Bc, Xc, dtc, cs, He, Dh)
                    - ((Cc * Bc).sum(1) * dtc)[:, None] * Xc),
    # the entry state read without its decay into the chunk
    "entry_undecayed": ("chunk_output", lambda Cc, Bc, Xc, dtc, cs, He, Dh: _CHUNK_OUTPUT(Cc, Bc, Xc, dtc, cs, He, Dh)
                        + (1.0 - np.exp(cs))[:, None] * (Cc @ He.T)),
    # the cumulative decay shifted by one token (exclusive instead of inclusive)
    "exclusive_cumsum": ("chunk_decay", lambda a: np.concatenate([[0.0], np.cumsum(a)[:-1]])),
}
_CHUNK_OUTPUT = oracle.chunk_output
_STATE_PASSING = oracle.state_passing


@pytest.mark.parametrize("name", sorted(PLANTED))
def test_chunked_planted_mistakes_are_caught(name, monkeypatch):
    step, fn = PLANTED[name]
    case = _rand_case(7, b=1, L=24, H=2, P=3, N=4, G=1)
    yr, fr = oracle.recurrent(**case)
    _planted(monkeypatch, step, fn)
    yc, fc = oracle.chunked(chunk=8, **case)
    assert max(_rel(yc, yr), _rel(fc, fr)) > 1e-3


# ---------------------------------------------------------------- one unit
# oracle.recurrent_unit checks the full-size workloads one (sequence, head) at
# a time and is the CPU baseline's timed code.  It slices the inputs down to
# one unit (the head's group, the sequence's row or packed range, its initial
# state) and runs the recurrence on them; the recurrence itself is pinned
# above, so what is pinned here is the slicing: every unit must equal, bit for
# bit, the same unit of one run over all the inputs.

def _unit_cases():
    return {
        # G > 1: heads 0-2 use group 0, heads 3-5 group 1, heads 6-8 group 2
        "groups": _rand_case(81, b=2, L=37, H=9, P=3, N=4, G=3),
        # packed sequences with initial states, an empty sequence in the middle
        "packed": _rand_case(82, b=1, L=50, H=4, P=2, N=3, G=2, cu=[0, 13, 13, 41, 50]),
        # no D, no initial states, one group per head
        "bare": _rand_case(83, b=3, L=20, H=2, P=3, N=2, G=2, init=False, D=False),
    }


def _unit_mismatches(unit_fn, c):
    """(s, h) units where unit_fn's result differs from the full run's."""
    y, fin = oracle.recurrent(**c)
    cu = c["cu_seqlens"]
    nseq = fin.shape[0]
    bad = []
    for s in range(nseq):
        for h in range(c["x"].shape[2]):
            yu, fu = unit_fn(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"],
                             c["initial_states"], cu, s, h)
            row, t0, t1 = (0, int(cu[s]), int(cu[s + 1])) if cu is not None else (s, 0, y.shape[1])
            if yu.shape != (t1 - t0, y.shape[3]) or not (
                    np.array_equal(yu, y[row, t0:t1, h]) and np.array_equal(fu, fin[s, h])):
                bad.append((s, h))
    return bad


@pytest.mark.parametrize("case", sorted(_unit_cases()))
def test_recurrent_unit_equals_slice_of_full_run(case):
    c = _unit_cases()[case]
    assert _unit_mismatches(oracle.recurrent_unit, c) == []


def test_recurrent_unit_empty_sequence_keeps_initial_state():
    c = _unit_cases()["packed"]
    yu, fu = oracle.recurrent_unit(c["x"], c["dt"], c["A"], c["B"], c["C"], c["D"],
                                   c["initial_states"], c["cu_seqlens"], 1, 2)
    assert yu.shape == (0, 2)
    np.testing.assert_array_equal(fu, c["initial_states"][1, 2].numpy())


def _unit_wrong_group(x, dt, A, B, C, D, S0, cu, s, h):
    # plausible slip: group h % G instead of h // (H / G)
    G = B.shape[2]
    sl = (lambda t, k: t[s:s + 1, :, k:k + 1]) if cu is None else \
        (lambda t, k: t[0:1, int(cu[s]):int(cu[s + 1]), k:k + 1])
    dts = dt[s:s + 1, :, h:h + 1] if cu is None else dt[0:1, int(cu[s]):int(cu[s + 1]), h:h + 1]
    y, fin = oracle.recurrent(sl(x, h), dts, A[h:h + 1], sl(B, h % G), sl(C, h % G),
                              None if D is None else D[h:h + 1],
                              None if S0 is None else S0[s:s + 1, h:h + 1], None)
    return y[0, :, 0, :], fin[0, 0]


def _unit_wrong_state_row(x, dt, A, B, C, D, S0, cu, s, h):
    # plausible slip: the initial state of sequence s taken from the batch row
    # (row 0 for every packed sequence)
    row = s if cu is None else 0
    S0r = None if S0 is None else S0[row:row + 1]
    return oracle.recurrent_unit(x, dt, A, B, C, D, S0r if S0 is None else
                                 S0r.expand(S0.shape[0], *S0.shape[1:]), cu, s, h)


def test_recurrent_unit_pin_catches_slicing_mistakes():
    cases = _unit_cases()
    assert _unit_mismatches(_unit_wrong_group, cases["groups"]) != []
    assert _unit_mismatches(_unit_wrong_state_row, cases["packed"]) != []
