"""The bench's roofline arithmetic, pinned to figures computed independently
from the workload shapes: the byte and FLOP counts of the 2.7B-shaped and
large-state layers (x, y, B, C, dt once each, plus the states; causal and
dense FLOP counts of the block decomposition), the fused kernel's split rule,
and the kernels one call launches (the gpu_launches figure)."""
import pytest

import bench


def _inp(batch, seqlen, nheads, headdim, dstate, ngroups, chunk=256, init=False):
    return dict(batch=batch, seqlen=seqlen, nheads=nheads, headdim=headdim, dstate=dstate,
                ngroups=ngroups, chunk=chunk, dtype="bf16", nseq=batch,
                initial_states=object() if init else None)


def test_cost_of_the_2p7b_shaped_layer():
    nbytes, causal, dense = bench.workload_cost(_inp(4, 8192, 80, 64, 128, 1))
    final_states = 4 * 80 * 64 * 128 * 4
    # x + y + B + C + dt (+ A, D): 698.35 MB; the final states are written once more
    assert nbytes - final_states == pytest.approx(698.35e6, abs=0.01e6)
    assert causal == pytest.approx(130.1e9, abs=0.05e9)
    # 32768 tokens x (80 (2.256.64 + 4.128.64) + 2.256.128) = 173.95e9, printed as 174.0
    assert dense == pytest.approx(174.0e9, abs=0.1e9)


def test_cost_of_the_large_state_layer():
    nbytes, causal, dense = bench.workload_cost(_inp(2, 16384, 32, 64, 256, 8, init=True))
    # initial and final states included
    assert nbytes == pytest.approx(549.45e6, abs=0.01e6)
    assert causal == pytest.approx(103.2e9, abs=0.05e9)
    assert dense == pytest.approx(137.4e9, abs=0.1e9)


def test_fused_split_rule_on_the_workloads():
    # 2.7B-shaped: 160 lanes, more than the SMs: one run; large state: 64 wide
    # lanes of 128 blocks: split; b2 L2048: 24 lanes of 16 blocks: split
    assert not bench.fused_splits_lanes(dict(_inp(4, 8192, 80, 64, 128, 1), cu_seqlens=None), 148)
    assert bench.fused_splits_lanes(dict(_inp(2, 16384, 32, 64, 256, 8), cu_seqlens=None), 148)
    assert bench.fused_splits_lanes(dict(_inp(2, 2048, 24, 64, 128, 1), cu_seqlens=None), 148)
    assert not bench.fused_splits_lanes(dict(_inp(2, 1024, 24, 64, 128, 1), cu_seqlens=None), 148)


def test_kernels_per_call_on_the_workloads():
    # the gpu_launches claim: one fused launch; a split call adds its
    # state-only pre run; packed sequences add the cu_seqlens check and the
    # lane-table set-up; the SIMT path runs k1-k4 (+ the check and k5 with
    # packing); the two-pass path its two kernels
    one = dict(_inp(4, 8192, 80, 64, 128, 1), cu_seqlens=None)
    split = dict(_inp(2, 16384, 32, 64, 256, 8), cu_seqlens=None)
    packed = dict(_inp(1, 32768, 64, 64, 128, 1), cu_seqlens=object())
    assert bench.launches_per_step("tc", one) == 1
    assert bench.launches_per_step("tc", split) == 2
    assert bench.launches_per_step("tc", packed) == 3
    assert bench.launches_per_step("simt", one) == 4
    assert bench.launches_per_step("simt", packed) == 6
    assert bench.launches_per_step("tc2", one) == 2
