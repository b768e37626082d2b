"""GPU parity of flp_logprob_entropy_k (K target tokens per scored row, the
K-candidate scoring that score centering trains on) against the float64
oracle, within |d logp|, |d ent| <= 1e-3.
"""
import numpy as np
import pytest
import torch

import entropy_tcgen05_vocab_gb300 as flp
import workloads
from oracle import coracle

pytestmark = pytest.mark.gpu
TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    flp.build()
    flp.lib()


def _candidates(T, V, K, seed):
    return torch.from_numpy(np.random.default_rng(seed).integers(0, V, size=(T, K)))


def _compare(d, tk, rows, tau, dtype="bf16"):
    logp, ent = flp.logprob_entropy_k(d["h"], d["W"], tk.cuda(), rows, tau)
    torch.cuda.synchronize()
    o = coracle.logprob_k(d["h"].cpu(), d["W"].cpu(), tk.numpy(),
                          None if rows is None else rows.cpu().numpy(), tau, dtype)
    assert np.abs(logp.cpu().double().numpy() - o["logp"]).max() <= TOL
    assert np.abs(ent.cpu().double().numpy() - o["ent"]).max() <= TOL
    return logp, ent


@pytest.mark.parametrize("K", [1, 2, 5, 8])
def test_k_targets_small(K):
    w = workloads.WORKLOADS[0].scaled(T=300, V=5001, seed=60 + K, w_std=0.05)
    d = workloads.make(w, device="cuda")
    _compare(d, _candidates(300, 5001, K, K), None, 0.7)


@pytest.mark.parametrize("n", [100, 128, 129])
def test_k_targets_both_sides_of_the_few_rows_switch(n):
    """n <= 128 scored rows run the single-CTA kernel, more the CTA pairs."""
    w = workloads.WORKLOADS[0].scaled(T=400, H=320, V=33000, seed=n + 3, w_std=0.05)
    d = workloads.make(w, device="cuda")
    rows = torch.from_numpy(workloads.sample_rows(400, n, seed=n)).cuda()
    _compare(d, _candidates(400, 33000, 6, n), rows, 0.8)


def test_k_targets_fp16_row_idx():
    w = workloads.WORKLOADS[2].scaled(T=2000, H=256, V=3000)
    d = workloads.make(w, device="cuda")
    _compare(d, _candidates(2000, 3000, 4, 61), d["row_idx"], 1.0, "fp16")


def test_single_candidate_equals_the_standard_op():
    d = workloads.make(0, device="cuda")
    lk, ek = flp.logprob_entropy_k(d["h"], d["W"], d["targets"][:, None], None, 1.0)
    l1, e1 = flp.logprob_entropy(d["h"], d["W"], d["targets"], None, 1.0)
    assert torch.equal(lk[:, 0], l1) and torch.equal(ek, e1)


def test_all_candidates_form_the_softmax():
    """K = V candidates: exp(logp) over them sums to 1."""
    w = workloads.WORKLOADS[0].scaled(T=130, H=64, V=8, seed=62, w_std=0.5)
    d = workloads.make(w, device="cuda")
    tk = torch.arange(8).repeat(130, 1)
    logp, _ = _compare(d, tk, None, 0.9)
    assert torch.allclose(logp.double().exp().sum(1).cpu(), torch.ones(130, dtype=torch.float64),
                          atol=1e-5)


def test_bad_candidates_are_nan_and_counted():
    w = workloads.WORKLOADS[0].scaled(T=200, V=1000, seed=63)
    d = workloads.make(w, device="cuda")
    tk = _candidates(200, 1000, 3, 63)
    tk[4, 1] = 1000
    tk[9, 2] = -5
    shape = flp.make_shape(200, 512, 1000, 200, torch.bfloat16)
    ws = torch.empty(flp.workspace_size(shape, flp.OP_LOGPROB_ENTROPY), dtype=torch.uint8,
                     device="cuda")
    logp, ent = flp.logprob_entropy_k(d["h"], d["W"], tk.cuda(), None, 1.0, workspace=ws)
    assert flp.read_device_status(ws)["bad_targets"] == 2
    lp = logp.cpu().numpy()
    assert np.isnan(lp[4, 1]) and np.isnan(lp[9, 2])
    assert np.isfinite(np.delete(lp.ravel(), [4 * 3 + 1, 9 * 3 + 2])).all()


def test_forward_scoring_workload_with_four_candidates_sampled():
    d = workloads.make(1, device="cuda")
    tk = _candidates(4096, d["workload"].V, 4, 64)
    tk[:, 0] = d["targets"].cpu()
    logp, ent = flp.logprob_entropy_k(d["h"], d["W"], tk.cuda(), None, d["tau"])
    torch.cuda.synchronize()
    pos = np.unique(np.concatenate([workloads.sample_rows(4096, 24, seed=65), [0, 4095]]))
    o = coracle.logprob_k(d["h"].cpu(), d["W"].cpu(), tk.numpy(), pos, d["tau"], "bf16")
    assert np.abs(logp.cpu().double().numpy()[pos] - o["logp"]).max() <= TOL
    assert np.abs(ent.cpu().double().numpy()[pos] - o["ent"]).max() <= TOL
