"""The entry points are CUDA-graph capturable: a captured forward, KL and
backward replay to the same bits as the eager calls.

Nothing in a call synchronises or allocates device memory (the workspace is
passed in), so a training step that calls the library can be captured once
and replayed.  Each call is made once eagerly first (that also caches the
tiling plan and the occupancy query), then captured and replayed on changed
inputs.
"""
import pytest
import torch

import entropy_tcgen05_vocab_gb300 as flp
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    flp.build()
    flp.lib()


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                                   # eager warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = fn()
    return g, out


def test_forward_and_backward_replay():
    w = workloads.WORKLOADS[4].scaled(T=600, H=256, V=5000, seed=91)
    d = workloads.make(w, device="cuda")
    n = d["n"]
    shape = flp.make_shape(w.T, w.H, w.V, n, torch.bfloat16)
    wsf = torch.empty(flp.workspace_size(shape, flp.OP_LOGPROB_ENTROPY), dtype=torch.uint8,
                      device="cuda")
    wsb = torch.empty(flp.workspace_size(shape, flp.OP_BACKWARD), dtype=torch.uint8, device="cuda")
    h = d["h"].clone()

    def step():
        logp, ent, lse, ez = flp.logprob_entropy(h, d["W"], d["targets"], d["row_idx"], d["tau"],
                                                 return_stats=True, workspace=wsf)
        dh, dW = flp.backward(h, d["W"], d["targets"], d["row_idx"], d["tau"], d["g1"], d["g2"],
                              lse, ez, workspace=wsb)
        return logp, ent, dh, dW

    g, out = _capture(step)
    for scale in (1.0, 0.5, 2.0):             # new inputs in the same buffers
        h.copy_((d["h"].float() * scale).to(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        ref = step()
        torch.cuda.synchronize()
        for a, b in zip(out, ref):
            assert torch.equal(a, b)


def test_kl_replay():
    w = workloads.WORKLOADS[3].scaled(T=500, H=256, V=6000, seed=92)
    d = workloads.make(w, device="cuda")
    shape = flp.make_shape(w.T, w.H, w.V, w.T, torch.bfloat16)
    ws = torch.empty(flp.workspace_size(shape, flp.OP_KL), dtype=torch.uint8, device="cuda")
    g, out = _capture(lambda: flp.kl_divergence(d["h_s"], d["W_s"], d["h_t"], d["W_t"],
                                                workspace=ws))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, flp.kl_divergence(d["h_s"], d["W_s"], d["h_t"], d["W_t"], workspace=ws))


def test_block_scaled_kl_replay():
    """The block-scaled KL (MXFP8 quantisation of the teacher rows, then the
    pipeline) captured and replayed on new teacher rows."""
    w = workloads.WORKLOADS[3].scaled(T=500, H=256, V=6000, seed=93)
    d = workloads.make(w, device="cuda")
    shape = flp.make_shape(w.T, w.H, w.V, w.T, torch.bfloat16)
    ws = torch.empty(flp.workspace_size(shape, flp.OP_KL_MX), dtype=torch.uint8, device="cuda")
    head = flp.mx_head_quantize(d["W_t"])
    h_t = d["h_t"].clone()
    g, out = _capture(lambda: flp.kl_divergence_mx(d["h_s"], d["W_s"], h_t, head, workspace=ws))
    for scale in (1.0, 0.5):
        h_t.copy_((d["h_t"].float() * scale).to(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, flp.kl_divergence_mx(d["h_s"], d["W_s"], h_t, head, workspace=ws))


def test_block_scaled_forward_replay():
    """The block-scaled forward (MXFP8 quantisation of the scored rows, then
    the pipeline) captured and replayed on new hidden rows."""
    w = workloads.WORKLOADS[1].scaled(T=600, H=256, V=7000, seed=94, targets="uniform")
    d = workloads.make(w, device="cuda")
    rows = torch.arange(0, 600, 3, device="cuda")
    shape = flp.make_shape(w.T, w.H, w.V, rows.numel(), torch.bfloat16)
    ws = torch.empty(flp.workspace_size(shape, flp.OP_LOGPROB_ENTROPY_MX), dtype=torch.uint8,
                     device="cuda")
    head = flp.mx_head_quantize(d["W"])
    h = d["h"].clone()
    g, out = _capture(lambda: flp.logprob_entropy_mx(h, head, w.V, d["targets"], rows, 0.7,
                                                     workspace=ws))
    for scale in (1.0, 0.5):
        h.copy_((d["h"].float() * scale).to(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        ref_out = flp.logprob_entropy_mx(h, head, w.V, d["targets"], rows, 0.7, workspace=ws)
        assert torch.equal(out[0], ref_out[0]) and torch.equal(out[1], ref_out[1])
