"""Sequence-parallel carry exchange, without a GPU.

* The composition in ``seqpar.ssd_scan_seqpar`` and its collective, on
  world_size 2 and 3 gloo ranks, with the oracle standing in for the three
  device steps: the oracle's recurrence scans each shard, the log-decay is
  summed in fp64, and the oracle's chunk-to-chunk state passing (pinned in
  test_oracle_pins.py) folds the gathered carries.  The shards' outputs
  concatenated and the final state must equal the oracle's unsharded
  recurrence to fp64 rounding; a fold that drops the shards' decay must not.
* The two C-ABI calls reject bad arguments on the host, before any device
  work, and their Python bindings check their inputs first.

QbitAI article "新架构Mamba更新二代！", section "Mamba-2：更强学习能力，更快训练推理"
(sequence parallelism).
"""
import ctypes
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
import ssd_synth

W0 = ssd_synth.Workload("seqpar_cpu", 2, 300, 3, 8, 16, 1, 64, "fp32", scale_bc=False)


class OracleOps:
    """The device steps of the exchange, computed by the oracle in fp64."""

    def __init__(self, plant=None):
        self.plant = plant

    def scan(self, x, dt, A, B, C, D, chunk_size, initial_states, out=None, final=True):
        y, fin = oracle.recurrent(x, dt, A, B, C, D, initial_states)
        return torch.from_numpy(y), torch.from_numpy(fin)

    def states(self, x, dt, A, B, C, chunk_size):
        return self.scan(x, dt, A, B, C, None, chunk_size, None)[1]

    def logdec(self, dt, A):
        a = dt.to(torch.float64) * A.to(torch.float64)          # (b, L, H)
        return a.sum(dim=1)

    def fold(self, S_all, ld_all, rank, initial_states):
        R, b, H, P, N = S_all.shape
        entry = np.zeros((b, H, P, N))
        final = np.zeros((b, H, P, N))
        for s in range(b):
            for h in range(H):
                S0 = (np.zeros((P, N)) if initial_states is None
                      else initial_states[s, h].to(torch.float64).numpy())
                decays = [0.0 if self.plant == "no_decay" else float(ld_all[q, s, h])
                          for q in range(R)]
                entries, fin = oracle.state_passing([S_all[q, s, h].numpy() for q in range(R)],
                                                    decays, S0)
                entry[s, h] = entries[rank]
                final[s, h] = fin
        return torch.from_numpy(entry), torch.from_numpy(final)

    def exchange(self, S, logdec, group):
        from mamba_ssd_layer_03_b300 import seqpar
        return seqpar.exchange_carries(S, logdec, group)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(seed, init):
    return ssd_synth.make_inputs(W0, seed=seed, init_states=init)


def _rank_main(rank, world, port, cuts, seed, init, plant, q):
    import torch.distributed as dist
    from mamba_ssd_layer_03_b300 import seqpar
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = _inputs(seed, init)
        t0, t1 = cuts[rank], cuts[rank + 1]
        sl = lambda t: t[:, t0:t1].contiguous()
        y, fin = seqpar.ssd_scan_seqpar(sl(inp["x"]), sl(inp["dt"]), inp["A"], sl(inp["B"]),
                                        sl(inp["C"]), inp["D"], W0.chunk,
                                        inp["initial_states"], ops=OracleOps(plant))
        q.put((rank, y.numpy(), fin.numpy()))
    finally:
        dist.destroy_process_group()


def _run_ranks(cuts, seed, init, plant=None):
    world = len(cuts) - 1
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, cuts, seed, init, plant, q))
             for r in range(world)]
    for p in procs:
        p.start()
    try:
        out = dict((r, (y, f)) for r, y, f in (q.get(timeout=180) for _ in range(world)))
    finally:
        for p in procs:
            p.join(timeout=60)
    for p in procs:
        assert p.exitcode == 0
    return out


@pytest.mark.parametrize("cuts,init", [
    ([0, 128, 300], True),            # two ranks, with initial states
    ([0, 77, 77, 300], False),        # three ranks, ragged, the middle one empty
])
def test_gloo_ranks_reproduce_the_unsharded_scan(cuts, init):
    out = _run_ranks(cuts, seed=5, init=init)
    inp = _inputs(5, init)
    y_ref, f_ref = oracle.recurrent(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                    inp["initial_states"])
    y = np.concatenate([out[r][0] for r in range(len(cuts) - 1)], axis=1)
    assert y.shape == y_ref.shape
    np.testing.assert_allclose(y, y_ref, rtol=1e-10, atol=1e-12)
    for r in out:
        np.testing.assert_allclose(out[r][1], f_ref, rtol=1e-10, atol=1e-12)


def test_gloo_ranks_catch_a_fold_without_decay():
    out = _run_ranks([0, 150, 300], seed=6, init=True, plant="no_decay")
    inp = _inputs(6, True)
    y_ref, _ = oracle.recurrent(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                inp["initial_states"])
    y1 = out[1][0]
    err = np.abs(y1 - y_ref[:, 150:]).max() / np.abs(y_ref).max()
    assert err > 1e-3


# ---------------------------------------------------------------- C ABI, host side

def _lib():
    import mamba_ssd_layer_03_b300 as ssd
    return ssd.load_library()


FAKE = ctypes.c_void_p(1 << 20)          # never dereferenced: checks come first
ODD = ctypes.c_void_p((1 << 20) + 2)     # not 4-byte aligned


def _fold(lib, nshards=2, rank=0, nseq=1, H=2, P=4, N=8, S=FAKE, ld=FAKE, init=None,
          entry=FAKE, final=None):
    return lib.ssd_seqpar_fold(nshards, rank, nseq, H, P, N, S, ld, init, entry, final, None)


@pytest.mark.parametrize("kw,code", [
    (dict(nshards=0), 1), (dict(rank=2), 1), (dict(rank=-1), 1), (dict(nseq=-1), 1),
    (dict(H=0), 1), (dict(P=0), 1), (dict(N=0), 1),
    (dict(S=None), 1), (dict(ld=None), 1), (dict(entry=None, final=None), 1),
    (dict(S=ODD), 2), (dict(init=ODD), 2), (dict(entry=ODD), 2), (dict(final=ODD), 2),
    (dict(nshards=1 << 20, nseq=1 << 20, H=1 << 10, P=1 << 10, N=1 << 10), 2),
    (dict(nseq=0, S=None, ld=None, entry=None), 0),
])
def test_fold_rejects_on_host(kw, code):
    assert _fold(_lib(), **kw) == code


def _logdec(lib, batch=2, seqlen=10, H=4, nseq=None, dt=FAKE, A=FAKE, out=FAKE, tf=None):
    import mamba_ssd_layer_03_b300 as ssd
    shape = ssd.make_shape(batch, seqlen, H, 1, 1, 1, 64, batch if nseq is None else nseq,
                           torch.float32, "simt")
    return lib.ssd_seqpar_logdec(ctypes.byref(shape), dt, tf, A, out, None)


def test_logdec_rejects_on_host():
    import mamba_ssd_layer_03_b300 as ssd
    lib = _lib()
    assert lib.ssd_seqpar_logdec(None, FAKE, None, FAKE, FAKE, None) == 1
    assert _logdec(lib, nseq=1) == 1                      # nseq must equal batch
    assert _logdec(lib, dt=None) == 1
    assert _logdec(lib, A=None) == 1
    assert _logdec(lib, out=None) == 1
    assert _logdec(lib, dt=ODD) == 2
    assert _logdec(lib, out=ODD) == 2
    assert _logdec(lib, seqlen=1 << 31) == 2
    bad = ssd.SsdDtTransform(None, 1, 1.0, 0.5)           # dt_min > dt_max
    assert _logdec(lib, tf=ctypes.byref(bad)) == 1
    odd_bias = ssd.SsdDtTransform((1 << 20) + 2, 1, 0.0, float("inf"))
    assert _logdec(lib, tf=ctypes.byref(odd_bias)) == 2
    assert _logdec(lib, batch=0, dt=None, A=None, out=None) == 0   # nothing to do
    assert _logdec(lib, seqlen=0, dt=None, A=None) == 1          # A still required


def test_python_bindings_check_inputs_first():
    from mamba_ssd_layer_03_b300 import seqpar
    dt = torch.rand(2, 10, 4)
    with pytest.raises(ValueError, match="CUDA"):
        seqpar.shard_logdec(dt, torch.rand(4))
    with pytest.raises(ValueError, match="shape"):
        seqpar.shard_logdec(dt, torch.rand(3))
    with pytest.raises(TypeError):
        seqpar.shard_logdec(dt.double(), torch.rand(4))
    S = torch.zeros(2, 1, 4, 2, 3)
    ld = torch.zeros(2, 1, 4)
    with pytest.raises(ValueError, match="outside"):
        seqpar.fold_carries(S, ld, 2)
    with pytest.raises(ValueError, match="shape"):
        seqpar.fold_carries(S, torch.zeros(2, 1, 3), 0)
    with pytest.raises(ValueError, match="CUDA"):
        seqpar.fold_carries(S, ld, 1)
