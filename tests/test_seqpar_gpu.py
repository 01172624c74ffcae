"""Sequence-parallel carry exchange on the GPU, against the fp64 oracle.

QbitAI article "新架构Mamba更新二代！", section "Mamba-2：更强学习能力，更快训练推理"
(sequence parallelism): a sequence cut into consecutive shards is scanned
shard by shard, each from a zero state; the shards' carries (end state and
total log-decay) are gathered and folded into every shard's entry state, and
each shard is scanned again from it.

* ``ssd_seqpar_logdec`` against the fp64 sum of dt' A (with and without the
  step-size transform), and ``ssd_seqpar_fold`` against the oracle's
  chunk-to-chunk state passing, which is the same recurrence over shards.
* The whole exchange through the library's kernels with the shards run one
  after another on one GPU (the gathered carries are a plain stack), for two
  to four shards (ragged, one empty), every scan path, with and without D,
  initial states and the transform: the shards' y and the final state
  against the oracle's unsharded recurrence.
* ``ssd_scan_seqpar`` end to end on two gloo ranks that share the GPU (the
  collective runs on the host: no kernel of one rank waits for the other).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
import ssd_synth
from parity_util import TOL, rel_err

pytestmark = pytest.mark.gpu

W_BF16 = ssd_synth.WORKLOADS[1]        # bf16, headdim 64, dstate 128, chunk 256
W_FP32 = ssd_synth.WORKLOADS[0]        # fp32, headdim 16, dstate 16, chunk 64


@pytest.mark.parametrize("transform", [False, True])
def test_logdec_matches_the_fp64_sum(transform):
    from mamba_ssd_layer_03_b300 import seqpar
    # 80 heads: two full 32-head blocks and a ragged one; L not a multiple of
    # the token stride
    inp = ssd_synth.make_inputs(ssd_synth.WORKLOADS[2], seed=41, batch=3, seqlen=3001)
    A = inp["A"]
    if transform:
        dt_in, tf = inp["dt_raw"], dict(dt_bias=inp["dt_bias"].cuda(), dt_softplus=True,
                                        dt_limit=(1e-3, 0.08))
        dt_ref = oracle.dt_transform(inp["dt_raw"], inp["dt_bias"], True, 1e-3, 0.08)
    else:
        dt_in, tf = inp["dt"], {}
        dt_ref = oracle._f64(inp["dt"])
    got = seqpar.shard_logdec(dt_in.cuda(), A.cuda(), **tf)
    torch.cuda.synchronize()
    ref = (dt_ref * oracle._f64(A)[None, None, :]).sum(axis=1)
    assert got.shape == (3, 80)
    np.testing.assert_allclose(got.cpu().numpy(), ref, rtol=1e-5, atol=0)


def test_logdec_of_an_empty_shard_is_zero():
    from mamba_ssd_layer_03_b300 import seqpar
    got = seqpar.shard_logdec(torch.zeros(2, 0, 5, device="cuda"), -torch.ones(5, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(got.cpu(), torch.zeros(2, 5))


@pytest.mark.parametrize("init", [False, True])
def test_fold_matches_oracle_state_passing(init):
    from mamba_ssd_layer_03_b300 import seqpar
    g = torch.Generator().manual_seed(42)
    R, b, H, P, N = 4, 2, 3, 16, 40
    S_all = torch.randn(R, b, H, P, N, generator=g)
    # decays from none (0) through moderate to total loss of the state (-200)
    ld_all = -torch.rand(R, b, H, generator=g) * 3.0
    ld_all[1, 0, 0], ld_all[2, 1, 2], ld_all[0, 1, 1] = 0.0, -200.0, -0.0
    S0 = torch.randn(b, H, P, N, generator=g) if init else None
    for rank in range(R):
        entry, final = seqpar.fold_carries(S_all.cuda(), ld_all.cuda(), rank,
                                           None if S0 is None else S0.cuda())
        torch.cuda.synchronize()
        for s in range(b):
            for h in range(H):
                z = np.zeros((P, N)) if S0 is None else S0[s, h].double().numpy()
                entries, fin = oracle.state_passing(
                    [S_all[q, s, h].double().numpy() for q in range(R)],
                    [float(ld_all[q, s, h]) for q in range(R)], z)
                np.testing.assert_allclose(entry[s, h].cpu().numpy(), entries[rank],
                                           rtol=1e-5, atol=1e-5)
                np.testing.assert_allclose(final[s, h].cpu().numpy(), fin, rtol=1e-5, atol=1e-5)


def _shards_on_one_gpu(inp, cuts, algo, D=True, init=True, tf=None):
    """The exchange with the shards run in turn on this GPU: every scan, the
    log-decay and the fold are the library's kernels; the all-gather is a
    stack of the shards' carries."""
    from mamba_ssd_layer_03_b300 import seqpar
    tf = tf or {}
    ops = seqpar.CudaOps(algo, **tf)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    dt = c["dt_raw"] if tf else c["dt"]
    sl = lambda t, r: t[:, cuts[r]:cuts[r + 1]].contiguous()
    R = len(cuts) - 1
    Dv = c["D"] if D else None
    S0 = c["initial_states"] if init else None
    carries, lds = [], []
    for r in range(R):
        _, S = ops.scan(sl(c["x"], r), sl(dt, r), c["A"], sl(c["B"], r), sl(c["C"], r), None,
                        inp["chunk"], None)
        carries.append(S)
        lds.append(ops.logdec(sl(dt, r), c["A"]))
    S_all, ld_all = torch.stack(carries), torch.stack(lds)
    ys, finals = [], []
    for r in range(R):
        entry, fin = ops.fold(S_all, ld_all, r, S0)
        y, _ = ops.scan(sl(c["x"], r), sl(dt, r), c["A"], sl(c["B"], r), sl(c["C"], r), Dv,
                        inp["chunk"], entry, final=False)
        ys.append(y)
        finals.append(fin)
    torch.cuda.synchronize()
    y = torch.cat(ys, dim=1).float().cpu().numpy()
    for f in finals[1:]:
        assert torch.equal(f, finals[0])
    return y, finals[0].cpu().numpy()


CUTS = {2: [0, 384, 1000], 3: [0, 300, 300, 1000], 4: [0, 1, 257, 700, 1000]}


@pytest.mark.parametrize("algo", ["tc", "tc2", "simt"])
@pytest.mark.parametrize("R", [2, 3, 4])
def test_bf16_shards_match_the_unsharded_oracle(algo, R):
    inp = ssd_synth.make_inputs(W_BF16, seed=43 + R, batch=2, seqlen=1000, nheads=8,
                                init_states=True)
    for D in (True, False):
        y, fin = _shards_on_one_gpu(inp, CUTS[R], algo, D=D)
        y_ref, f_ref = oracle.recurrent(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                                        inp["D"] if D else None, inp["initial_states"])
        assert rel_err(y, y_ref) <= TOL["bf16"], (D, rel_err(y, y_ref))
        assert rel_err(fin, f_ref) <= TOL["bf16"], (D, rel_err(fin, f_ref))


def test_bf16_shards_with_the_step_size_transform():
    inp = ssd_synth.make_inputs(W_BF16, seed=47, batch=2, seqlen=1000, nheads=8)
    tf = dict(dt_bias=inp["dt_bias"].cuda(), dt_softplus=True, dt_limit=(1e-3, 0.08))
    y, fin = _shards_on_one_gpu(inp, CUTS[3], "tc", D=False, init=False, tf=tf)
    dt_ref = oracle.dt_transform(inp["dt_raw"], inp["dt_bias"], True, 1e-3, 0.08)
    y_ref, f_ref = oracle.recurrent(inp["x"], dt_ref, inp["A"], inp["B"], inp["C"])
    assert rel_err(y, y_ref) <= TOL["bf16"]
    assert rel_err(fin, f_ref) <= TOL["bf16"]


@pytest.mark.parametrize("R", [2, 3])
def test_fp32_shards_match_the_unsharded_oracle(R):
    inp = ssd_synth.make_inputs(W_FP32, seed=48 + R, batch=2, seqlen=1000, init_states=True)
    y, fin = _shards_on_one_gpu(inp, CUTS[R], "simt", D=False)
    y_ref, f_ref = oracle.recurrent(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], None,
                                    inp["initial_states"])
    assert rel_err(y, y_ref) <= TOL["fp32"]
    assert rel_err(fin, f_ref) <= TOL["fp32"]


# ------------------------------------------------- two gloo ranks sharing one GPU

def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _gpu_rank_main(rank, world, port, cuts, q):
    import torch.distributed as dist
    from mamba_ssd_layer_03_b300 import seqpar

    class HostGatherOps(seqpar.CudaOps):
        # gloo gathers host tensors: stage the carries through the host
        def exchange(self, S, logdec, group):
            S_all, ld_all = seqpar.exchange_carries(S.cpu(), logdec.cpu(), group)
            return S_all.to(S.device), ld_all.to(logdec.device)

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = ssd_synth.make_inputs(W_BF16, seed=49, batch=2, seqlen=1000, nheads=8,
                                    init_states=True)
        c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        sl = lambda t: t[:, cuts[rank]:cuts[rank + 1]].contiguous()
        y, fin = seqpar.ssd_scan_seqpar(sl(c["x"]), sl(c["dt"]), c["A"], sl(c["B"]), sl(c["C"]),
                                        c["D"], W_BF16.chunk, c["initial_states"],
                                        ops=HostGatherOps("auto"))
        torch.cuda.synchronize()
        q.put((rank, y.float().cpu().numpy(), fin.cpu().numpy()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_on_one_gpu_end_to_end():
    cuts = [0, 512, 1000]
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_gpu_rank_main, args=(r, world, port, cuts, q))
             for r in range(world)]
    for p in procs:
        p.start()
    try:
        out = dict((r, (y, f)) for r, y, f in (q.get(timeout=300) for _ in range(world)))
    finally:
        for p in procs:
            p.join(timeout=120)
    for p in procs:
        assert p.exitcode == 0
    inp = ssd_synth.make_inputs(W_BF16, seed=49, batch=2, seqlen=1000, nheads=8,
                                init_states=True)
    y_ref, f_ref = oracle.recurrent(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                    inp["initial_states"])
    y = np.concatenate([out[0][0], out[1][0]], axis=1)
    assert rel_err(y, y_ref) <= TOL["bf16"]
    for r in (0, 1):
        assert rel_err(out[r][1], f_ref) <= TOL["bf16"]
