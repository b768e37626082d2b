"""GPU parity of flp_logprob_entropy against the float64 oracle.

Element by element on small cases that still span several 128-row tiles,
several 256-column vocabulary tiles and ragged tails in rows, vocabulary and
hidden size; on seeded row samples at the full sizes of the forward-scoring
(4096 x 4096 x 151,936, tau 0.7) and long-packed (49,152 packed, H 5120,
V 38,016, fp16) workloads, in the same launch configuration the bench times:
512 seeded rows plus the first and last rows, the rows with the most negative
log-probs and those with the lowest and highest entropies.
Tolerance: |d logp|, |d ent| <= 1e-3 absolute on every checked row.
"""
import math

import numpy as np
import pytest
import torch

import entropy_tcgen05_vocab_gb300 as flp
import workloads
from oracle import coracle, ref

pytestmark = pytest.mark.gpu
TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    flp.build()
    flp.lib()


def _dt(dtype):
    return "bf16" if dtype == torch.bfloat16 else "fp16"


def _check(got, want, what, tol=TOL):
    got = got.detach().cpu().double().numpy()
    err = np.abs(got - want)
    assert np.all(np.isfinite(got)), what + ": non-finite output"
    assert err.max() <= tol, "%s: max |diff| %.3e at %d" % (what, err.max(), int(err.argmax()))
    return float(err.max())


def _run_and_compare(h, W, targets, row_idx, tau, oracle="c"):
    logp, ent, lse, ez = flp.logprob_entropy(h, W, targets, row_idx, tau, return_stats=True)
    torch.cuda.synchronize()
    rows = None if row_idx is None else row_idx.cpu().numpy()
    f = coracle.logprob_entropy if oracle == "c" else ref.logprob_entropy
    o = f(h.cpu(), W.cpu(), targets.cpu().numpy(), rows, tau, _dt(h.dtype))
    _check(logp, o["logp"], "logp")
    _check(ent, o["ent"], "ent")
    _check(lse, o["lse"], "lse")
    _check(ez, o["ez"], "ez", tol=2e-3)
    return logp, ent


def test_tiny_workload_full():
    d = workloads.make(0, device="cuda")
    _run_and_compare(d["h"], d["W"], d["targets"], None, 1.0)


@pytest.mark.parametrize("tau", [0.7, 1.0, 2.5])
def test_temperatures(tau):
    w = workloads.WORKLOADS[0].scaled(T=300, V=5000, seed=21, w_std=0.05)
    d = workloads.make(w, device="cuda")
    _run_and_compare(d["h"], d["W"], d["targets"], None, tau)


@pytest.mark.parametrize("T,H,V", [
    (129, 64, 256),      # one row past a tile; one vocabulary tile exactly
    (200, 520, 8000),    # H not a multiple of 64; last vocab tile 64 columns
    (384, 256, 8200),    # last vocab tile 8 columns
    (1, 8, 8),           # single row, minimal hidden size, V inside one 32-column chunk
    (40, 96, 33),        # V one past a 32-column chunk
    (1000, 128, 20000),  # many row tiles and vocab tiles
])
def test_ragged_shapes(T, H, V):
    w = workloads.WORKLOADS[0].scaled(T=T, H=H, V=V, seed=T + H + V, w_std=0.08)
    d = workloads.make(w, device="cuda")
    _run_and_compare(d["h"], d["W"], d["targets"], None, 0.7)


def test_fp16_packed_rows():
    w = workloads.WORKLOADS[2].scaled(T=3000, H=256, V=6000)
    d = workloads.make(w, device="cuda")
    assert d["h"].dtype == torch.float16
    _run_and_compare(d["h"], d["W"], d["targets"], d["row_idx"], 1.0)


def test_row_idx_unsorted_with_duplicates():
    w = workloads.WORKLOADS[0].scaled(T=500, V=3000, seed=22)
    d = workloads.make(w, device="cuda")
    rows = torch.tensor([499, 3, 3, 250, 0, 17, 499, 128, 127], device="cuda")
    _run_and_compare(d["h"], d["W"], d["targets"], rows, 0.9)


def test_strided_hidden_and_weight():
    w = workloads.WORKLOADS[0].scaled(T=260, H=192, V=4100, seed=23)
    d = workloads.make(w, device="cuda")
    hb = torch.zeros(260, 256, dtype=torch.bfloat16, device="cuda")
    Wb = torch.zeros(4100, 200, dtype=torch.bfloat16, device="cuda")
    hb[:, :192] = d["h"]
    Wb[:, :192] = d["W"]
    h, W = hb[:, :192], Wb[:, :192]
    assert h.stride(0) == 256 and W.stride(0) == 200
    logp, ent = flp.logprob_entropy(h, W, d["targets"], None, 1.0)
    o = coracle.logprob_entropy(d["h"].cpu(), d["W"].cpu(), d["targets"].cpu(), None, 1.0, "bf16")
    _check(logp, o["logp"], "logp")
    _check(ent, o["ent"], "ent")


def test_zero_weight_closed_form():
    h = torch.randn(300, 128, device="cuda").to(torch.bfloat16)
    W = torch.zeros(10000, 128, dtype=torch.bfloat16, device="cuda")
    t = torch.randint(0, 10000, (300,), device="cuda")
    for tau in (0.7, 1.0):
        logp, ent = flp.logprob_entropy(h, W, t, None, tau)
        _check(logp, np.full(300, -math.log(10000)), "logp", tol=1e-5)
        _check(ent, np.full(300, math.log(10000)), "ent", tol=1e-5)


def test_one_hot_dominant_rows():
    g = torch.Generator().manual_seed(24)
    H, V, T = 64, 3000, 130
    h = torch.randn(T, H, generator=g, dtype=torch.float64)
    W = torch.randn(V, H, generator=g, dtype=torch.float64) * 0.01
    tg = torch.randint(0, V, (T,), generator=g)
    for i in range(0, T, 13):   # rows sharing no target
        W[tg[i]] = 70.0 * h[i] / (h[i] @ h[i])
    hb, Wb = h.to(torch.bfloat16), W.to(torch.bfloat16)
    rows = torch.arange(0, T, 13)
    logp, ent = flp.logprob_entropy(hb.cuda(), Wb.cuda(), tg.cuda(), rows.cuda(), 1.0)
    o = coracle.logprob_entropy(hb, Wb, tg.numpy(), rows.numpy(), 1.0, "bf16")
    assert np.all(o["logp"] > -1e-10)
    _check(logp, o["logp"], "logp")
    _check(ent, o["ent"], "ent")


@pytest.mark.parametrize("tau", [0.1, 10.0, 50.0])
def test_extreme_temperatures(tau):
    """Sharp (logits / 0.1 spread over tens of nats) and nearly flat (entropy
    close to ln V) distributions."""
    w = workloads.WORKLOADS[0].scaled(T=300, V=5000, seed=26, w_std=0.05)
    d = workloads.make(w, device="cuda")
    logp, ent = _run_and_compare(d["h"], d["W"], d["targets"], None, tau)
    if tau >= 10.0:
        assert np.all(ent.cpu().numpy() > math.log(5000) - 0.1)


def test_large_logits():
    """Hidden states 30x the recipe's scale: logits in the hundreds, so the
    running max moves by large steps and almost all the mass sits on a few
    tokens per row."""
    w = workloads.WORKLOADS[0].scaled(T=260, V=7000, seed=27, w_std=0.05, h_std=30.0)
    d = workloads.make(w, device="cuda")
    _run_and_compare(d["h"], d["W"], d["targets"], None, 1.0)


def test_single_token_vocabulary():
    """V = 1: every row's distribution is the one token, logp = 0, entropy 0
    (up to FP32 rounding: the fold works in base 2, so z/tau and the LSE
    reach the same value by different roundings)."""
    w = workloads.WORKLOADS[0].scaled(T=200, H=64, V=1, seed=28)
    d = workloads.make(w, device="cuda")
    logp, ent = _run_and_compare(d["h"], d["W"], d["targets"], None, 0.7)
    assert logp.abs().max().item() <= 1e-6 and ent.abs().max().item() <= 1e-6


def test_no_scored_rows():
    d = workloads.make(workloads.WORKLOADS[0].scaled(T=64, V=512), device="cuda")
    rows = torch.zeros(0, dtype=torch.int64, device="cuda")
    logp, ent = flp.logprob_entropy(d["h"], d["W"], d["targets"], rows, 1.0)
    assert logp.numel() == 0 and ent.numel() == 0


def test_bad_targets_and_rows_are_nan_and_counted():
    w = workloads.WORKLOADS[0].scaled(T=300, V=2000, seed=25)
    d = workloads.make(w, device="cuda")
    tg = d["targets"].clone()
    tg[5] = 2000
    tg[7] = -3
    rows = torch.tensor([5, 6, 7, 300, -1, 8], device="cuda")
    shape = flp.make_shape(300, 512, 2000, 6, torch.bfloat16)
    ws = torch.empty(flp.workspace_size(shape, flp.OP_LOGPROB_ENTROPY), dtype=torch.uint8,
                     device="cuda")
    logp, ent = flp.logprob_entropy(d["h"], d["W"], tg, rows, 1.0, workspace=ws)
    st = flp.read_device_status(ws)
    assert st == {"bad_targets": 2, "bad_rows": 2, "timeouts": 0, "empty_supports": 0}
    lp, en = logp.cpu().numpy(), ent.cpu().numpy()
    assert np.isnan(lp[[0, 2, 3, 4]]).all() and np.isfinite(lp[[1, 5]]).all()
    assert np.isfinite(en[[0, 1, 2, 5]]).all() and np.isnan(en[[3, 4]]).all()
    o = coracle.logprob_entropy(d["h"].cpu(), d["W"].cpu(), tg.cpu().numpy(),
                                np.array([6, 8, 5]), 1.0, "bf16")
    _check(logp[[1, 5]], o["logp"][:2], "logp")
    _check(ent[[1, 5, 0]], o["ent"], "ent")


def test_repeated_calls_are_deterministic():
    d = workloads.make(0, device="cuda")
    a = flp.logprob_entropy(d["h"], d["W"], d["targets"], None, 1.0)
    b = flp.logprob_entropy(d["h"], d["W"], d["targets"], None, 1.0)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# ---------------------------------------------------------------- full sizes

def _extreme_rows(logp, ent, k=8):
    """Positions of the rows with the most negative log-prob (the target's
    logit furthest below the row's maximum) and the lowest and highest
    entropies: where the fold's precision is tested hardest."""
    lp, en = logp.detach().cpu().numpy(), ent.detach().cpu().numpy()
    return np.concatenate([np.argsort(lp)[:k], np.argsort(en)[:k // 2], np.argsort(en)[-(k // 2):]])


def _full_size(wid, k=512):
    d = workloads.make(wid, device="cuda")
    logp, ent = flp.logprob_entropy(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"])
    torch.cuda.synchronize()
    n = d["n"]
    pos = workloads.sample_rows(n, k, seed=wid)
    pos = np.unique(np.concatenate([pos, [0, n - 1], _extreme_rows(logp, ent)]))
    rows = pos if d["row_idx"] is None else d["row_idx"].cpu().numpy()[pos]
    o = ref.logprob_entropy(d["h"].cpu(), d["W"].cpu(), d["targets"].cpu().numpy(), rows,
                            d["tau"], d["workload"].dtype)
    e1 = _check(logp[torch.from_numpy(pos).cuda()], o["logp"], "logp")
    e2 = _check(ent[torch.from_numpy(pos).cuda()], o["ent"], "ent")
    # properties over every row
    lp, en = logp.cpu().numpy(), ent.cpu().numpy()
    assert np.all(np.isfinite(lp)) and np.all(lp <= 1e-4)
    assert np.all(en >= -1e-4) and np.all(en <= math.log(d["workload"].V) + 1e-4)
    print("workload %d: %d sampled rows, max|dlogp| %.2e, max|dent| %.2e" % (wid, len(pos), e1, e2))


def test_forward_scoring_workload_sampled():
    _full_size(1)


def test_long_packed_workload_sampled():
    _full_size(2)


@pytest.mark.parametrize("T,H,V", [
    (100, 2048, 262144),   # one row tile, 512 vocabulary tiles: the most splits
    (20000, 128, 512),     # 79 row tiles, one vocabulary tile
    (3000, 8192, 1000),    # long contraction, V inside two 512-column tiles
])
def test_planner_extremes(T, H, V):
    w = workloads.WORKLOADS[0].scaled(T=T, H=H, V=V, seed=T + V, w_std=0.03)
    d = workloads.make(w, device="cuda")
    rows = None
    if T > 1000:   # oracle on a sample of rows, outputs compared there
        rows = torch.from_numpy(workloads.sample_rows(T, 300, seed=7)).cuda()
    _run_and_compare(d["h"], d["W"], d["targets"], rows, 0.8)


@pytest.mark.parametrize("n", [1, 127, 128, 129])
def test_few_rows_path_boundary(n):
    """n <= 128 scored rows run single CTAs on 128 x 256 tiles, n > 128 CTA
    pairs; both sides of the switch, with a gather, against the oracle."""
    w = workloads.WORKLOADS[0].scaled(T=400, H=320, V=33000, seed=n, w_std=0.05)
    d = workloads.make(w, device="cuda")
    rows = torch.from_numpy(workloads.sample_rows(400, n, seed=n + 1)).cuda()
    plan = flp.plan(flp.make_shape(400, 320, 33000, n, torch.bfloat16), flp.OP_LOGPROB_ENTROPY, 152)
    assert plan["cta_group"] == (1 if n <= 128 else 2)
    _run_and_compare(d["h"], d["W"], d["targets"], rows, 0.8)


def test_kl_at_the_planner_extremes():
    w = workloads.WORKLOADS[3].scaled(T=64, H=1024, V=131072, seed=51)
    d = workloads.make(w, device="cuda")
    kl = flp.kl_divergence(d["h_s"], d["W_s"], d["h_t"], d["W_t"])
    want = coracle.kl(d["h_s"].cpu(), d["W_s"].cpu(), d["h_t"].cpu(), d["W_t"].cpu(), None, "bf16")
    _check(kl, want, "kl")


def test_no_vocabulary_sized_buffer_is_allocated():
    """The call allocates nothing beyond its outputs: the peak of torch's
    allocator over the call, with the workspace passed in, is the two [n]
    outputs, and the device's free memory is unchanged afterwards (the
    library itself never allocates).  The workspace is far below the [T, V]
    FP32 logits (2.5 GB at this size)."""
    d = workloads.make(1, device="cuda")
    w = d["workload"]
    shape = flp.make_shape(w.T, w.H, w.V, d["n"], torch.bfloat16)
    ws = torch.empty(flp.workspace_size(shape, flp.OP_LOGPROB_ENTROPY), dtype=torch.uint8,
                     device="cuda")
    flp.logprob_entropy(d["h"], d["W"], d["targets"], None, d["tau"], workspace=ws)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    logp, ent = flp.logprob_entropy(d["h"], d["W"], d["targets"], None, d["tau"], workspace=ws)
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated() - base
    assert peak <= 2 * 4 * w.T + (1 << 20), peak
    assert torch.cuda.mem_get_info()[0] >= free0 - (2 << 20)
    logits_bytes = w.T * w.V * 4
    assert ws.numel() * 20 < logits_bytes, (ws.numel(), logits_bytes)
    del logp, ent
