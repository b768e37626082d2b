"""Failure handling on the GPU without faulting it.

Every wait in the pipeline kernels is bounded.  A self-test kernel makes one
such wait run out (an mbarrier that nothing arrives on, 50 ms limit): the
wait must end, the timeout must be counted in the status the host reads, and
the context must stay usable for a normal call afterwards.  No trap, assert,
bad address or endless loop is involved.
"""
import numpy as np
import pytest
import torch

import entropy_tcgen05_vocab_gb300 as flp
import workloads
from oracle import coracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    flp.build()
    flp.lib()


def test_stalled_wait_is_reported_and_the_context_survives():
    st = flp.selftest_wait_timeout(50_000_000)
    assert st == {"bad_targets": 0, "bad_rows": 0, "timeouts": 1,
                  "empty_supports": 0}
    d = workloads.make(0, device="cuda")
    logp, ent = flp.logprob_entropy(d["h"], d["W"], d["targets"], None, 1.0)
    o = coracle.logprob_entropy(d["h"].cpu(), d["W"].cpu(), d["targets"].cpu(), None, 1.0, "bf16")
    assert np.abs(logp.cpu().double().numpy() - o["logp"]).max() <= 1e-3
    assert np.abs(ent.cpu().double().numpy() - o["ent"]).max() <= 1e-3


def test_normal_calls_report_no_timeouts():
    d = workloads.make(workloads.WORKLOADS[3].scaled(T=300, H=256, V=5000), device="cuda")
    shape = flp.make_shape(300, 256, 5000, 300, torch.bfloat16)
    ws = torch.empty(flp.workspace_size(shape, flp.OP_KL), dtype=torch.uint8, device="cuda")
    flp.kl_divergence(d["h_s"], d["W_s"], d["h_t"], d["W_t"], None, workspace=ws)
    assert flp.read_device_status(ws) == {"bad_targets": 0, "bad_rows": 0, "timeouts": 0,
                                          "empty_supports": 0}
