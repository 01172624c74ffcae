"""Failure detection on the GPU without a fault: one of the kernels' bounded
waits is made to run out (an mbarrier nothing completes, a handoff flag nothing
sets); the device must record SSD_ERR_DEVICE_TIMEOUT in the status word, the
call must return, and the context must stay usable for a normal scan."""
import pytest
import torch

import ssd_synth
from parity_util import TOL, oracle_full, rel_err, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("which", [0, 1], ids=["mbarrier", "handoff_flag"])
def test_bounded_wait_gives_up_and_reports(which):
    import mamba_ssd_layer_03_b300 as ssd
    assert ssd.selftest_wait_timeout(which) == 5   # SSD_ERR_DEVICE_TIMEOUT
    # the context is still usable: a normal scan runs and is correct
    inp = ssd_synth.make_inputs(ssd_synth.WORKLOADS[1], seed=51, batch=1, seqlen=300, nheads=4)
    y, fin = run_gpu(inp, algo="tc")
    y_ref, fin_ref = oracle_full(inp)
    assert rel_err(y, y_ref) <= TOL["bf16"]
    assert rel_err(fin, fin_ref) <= TOL["bf16"]
