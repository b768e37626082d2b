"""Failure handling on the GPU without faulting it.

Every wait in the pipeline kernels is bounded.  A self-test kernel makes one
such wait run out (an mbarrier that nothing arrives on, 50 ms limit): the
wait must end, the timeout must be counted in the status the host reads, and
the context must stay usable for a normal call afterwards.

The real pipelines' give-up path is driven the same way: flp_set_wait_limit
lowers the limit of their waits to 1 us, shorter than one tile of MMAs, so
the epilogue's wait for its first accumulator (and others) runs out.  The
kernels must then set their abort flag, let the copies and MMAs in flight
finish, free tensor memory and end; the call's status must count the
timeouts; and the next call with the default limit, on the same context,
must match the oracle.  The outputs of the timed-out call are not looked at.
No trap, assert, bad address or endless loop is involved.
"""
import numpy as np
import pytest
import torch

import entropy_tcgen05_vocab_gb300 as flp
import workloads
from oracle import coracle, ref

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


SHORT_NS = 1000     # 1 us
# H = 2048 (32 k-blocks): a CTA's first accumulator tile takes well over
# 1 us of MMAs whatever the granularity of the GPU's global timer, so the
# epilogue's wait for it runs out in every pipeline.
ABORT_H = 2048


class _ShortWaits:
    """Every call inside the block runs its kernels with 1 us waits."""

    def __enter__(self):
        flp.set_wait_limit(SHORT_NS)

    def __exit__(self, *exc):
        flp.set_wait_limit(0)


def _ws(T, H, V, n, op):
    shape = flp.make_shape(T, H, V, n, torch.bfloat16)
    return torch.empty(flp.workspace_size(shape, op), dtype=torch.uint8, device="cuda")


def _fwd_case():
    return workloads.make(workloads.WORKLOADS[0].scaled(H=ABORT_H), device="cuda")


def _forward_matches_oracle(d, rows=None):
    logp, ent = flp.logprob_entropy(d["h"], d["W"], d["targets"], rows, 1.0)
    o = coracle.logprob_entropy(d["h"].cpu(), d["W"].cpu(), d["targets"].cpu(),
                                None if rows is None else rows.cpu().numpy(), 1.0, "bf16")
    assert np.abs(logp.cpu().double().numpy() - o["logp"]).max() <= 1e-3
    assert np.abs(ent.cpu().double().numpy() - o["ent"]).max() <= 1e-3


@pytest.mark.parametrize("n", [256, 100])       # CTA pairs; the single-CTA few-rows path
def test_forward_pipeline_wait_that_runs_out_unwinds(n):
    d = _fwd_case()
    rows = None if n == 256 else torch.arange(n, device="cuda") * 2
    ws = _ws(256, ABORT_H, 8192, n, flp.OP_LOGPROB_ENTROPY)
    with _ShortWaits():
        flp.logprob_entropy(d["h"], d["W"], d["targets"], rows, 1.0, workspace=ws)
        st = flp.read_device_status(ws)
    assert st["timeouts"] > 0, st
    # the same workspace and context, default limit: a clean, correct call
    flp.logprob_entropy(d["h"], d["W"], d["targets"], rows, 1.0, workspace=ws)
    assert flp.read_device_status(ws)["timeouts"] == 0
    _forward_matches_oracle(d, rows)


@pytest.mark.parametrize("teacher", ["bf16", "mxfp4"])
def test_kl_pipeline_wait_that_runs_out_unwinds(teacher):
    k = workloads.make(workloads.WORKLOADS[3].scaled(T=256, H=ABORT_H, V=8192, seed=5),
                       device="cuda")
    ws = _ws(256, ABORT_H, 8192, 256, flp.OP_KL)
    if teacher == "mxfp4":
        packed, scales = flp.mxfp4_quantize(k["W_t"])
        run = lambda: flp.kl_divergence_mxfp4(k["h_s"], k["W_s"], k["h_t"], packed, scales,
                                              workspace=ws)
        opacked, oscales = coracle.mxfp4_quantize(k["W_t"].cpu(), "bf16")
        want = ref.kl_mxfp4(k["h_s"].cpu(), k["W_s"].cpu(), k["h_t"].cpu(), opacked, oscales, None,
                            "bf16")
    else:
        run = lambda: flp.kl_divergence(k["h_s"], k["W_s"], k["h_t"], k["W_t"], workspace=ws)
        want = coracle.kl(k["h_s"].cpu(), k["W_s"].cpu(), k["h_t"].cpu(), k["W_t"].cpu(), None,
                          "bf16")
    with _ShortWaits():
        run()
        st = flp.read_device_status(ws)
    assert st["timeouts"] > 0, st
    kl = run()
    assert flp.read_device_status(ws)["timeouts"] == 0
    assert np.abs(kl.cpu().double().numpy() - want).max() <= 1e-3


def test_backward_pipelines_wait_that_runs_out_unwinds():
    """The statistics pass, the gradient pass and the dh and dW GEMMs all run
    with 1 us waits; each gives up and unwinds."""
    b = workloads.make(workloads.WORKLOADS[4].scaled(T=300, H=ABORT_H, V=4000, seed=6),
                       device="cuda")
    shape = flp.make_shape(300, ABORT_H, 4000, b["n"], torch.bfloat16)
    ws = torch.empty(flp.workspace_size(shape, flp.OP_BACKWARD), dtype=torch.uint8,
                     device="cuda")
    args = (b["h"], b["W"], b["targets"], b["row_idx"], b["tau"], b["g1"], b["g2"])
    with _ShortWaits():
        flp.backward(*args, workspace=ws)
        st = flp.read_device_status(ws)
    assert st["timeouts"] > 0, st
    dh, dW = flp.backward(*args, workspace=ws)
    assert flp.read_device_status(ws)["timeouts"] == 0
    rows = b["row_idx"].cpu().numpy()
    dh_rows, dW_ref = coracle.backward(b["h"].cpu(), b["W"].cpu(), b["targets"].cpu().numpy(),
                                       rows, b["tau"], b["g1"].cpu().numpy(),
                                       b["g2"].cpu().numpy(), "bf16")
    dh_ref = coracle.scatter_rows(dh_rows, rows, b["h"].shape[0])
    for got, want in ((dh, dh_ref), (dW, dW_ref)):
        g = got.cpu().double().numpy()
        assert np.linalg.norm(g - want) <= 1e-2 * np.linalg.norm(want)


def test_block_scaled_kl_pipeline_wait_that_runs_out_unwinds():
    """The two-ring pipeline of flp_kl_mx (student and teacher rings, scale
    copies into TMEM) gives up, drains and frees its TMEM the same way."""
    k = workloads.make(workloads.WORKLOADS[3].scaled(T=256, H=ABORT_H, V=8192, seed=5),
                       device="cuda")
    ws = _ws(256, ABORT_H, 8192, 256, flp.OP_KL_MX)
    head = flp.mx_head_quantize(k["W_t"])
    run = lambda: flp.kl_divergence_mx(k["h_s"], k["W_s"], k["h_t"], head, workspace=ws)
    packed, scales = coracle.mxfp4_quantize(k["W_t"].cpu(), "bf16")
    want = coracle.kl_mx(k["h_s"].cpu(), k["W_s"].cpu(), k["h_t"].cpu(), packed, scales, None,
                         "bf16")
    with _ShortWaits():
        run()
        st = flp.read_device_status(ws)
    assert st["timeouts"] > 0, st
    kl = run()
    assert flp.read_device_status(ws)["timeouts"] == 0
    assert np.abs(kl.cpu().double().numpy() - want).max() <= 1e-3


def test_block_scaled_forward_pipeline_wait_that_runs_out_unwinds():
    """The block-scaled forward (one ring, scale slots fewer than its stages)
    gives up, drains and frees its TMEM the same way."""
    d = _fwd_case()
    V = 8192
    ws = _ws(256, ABORT_H, V, 256, flp.OP_LOGPROB_ENTROPY_MX)
    head = flp.mx_head_quantize(d["W"])
    run = lambda: flp.logprob_entropy_mx(d["h"], head, V, d["targets"], None, 1.0, workspace=ws)
    packed, scales = coracle.mxfp4_quantize(d["W"].cpu(), "bf16")
    want = coracle.logprob_entropy_mx(d["h"].cpu(), packed, scales, V, d["targets"].cpu().numpy(),
                                      None, 1.0, "bf16")
    with _ShortWaits():
        run()
        st = flp.read_device_status(ws)
    assert st["timeouts"] > 0, st
    logp, ent = run()
    assert flp.read_device_status(ws)["timeouts"] == 0
    assert np.abs(logp.cpu().double().numpy() - want["logp"]).max() <= 1e-3
    assert np.abs(ent.cpu().double().numpy() - want["ent"]).max() <= 1e-3
