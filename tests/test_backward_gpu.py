"""GPU parity of flp_backward (dL/dh, dL/dW of sum g1 logp + g2 ent) against
the float64 oracle.

Tolerance (per tensor): ||d - ref||_F <= 1e-2 ||ref||_F, and every element
within 1e-2 max|ref|.  Small cases compare dh and dW in full, across several
row and vocabulary tiles, ragged hidden and vocabulary sizes, fp16, several
row chunks and caller-supplied statistics.  At the full backward workload
(16,384 rows, 60 % scored, H 4096, V 151,936) the oracle first computes
every scored row's statistics (log-sum-exp and E[z'], a float64 pass over
the whole vocabulary, which every element of dW depends on); then dh is
compared on 512 sampled rows and the rows with the most negative log-probs,
and dW element by element on 256 sampled vocabulary rows plus the targets of
those worst rows and the last row.  dW is also checked through a property
that holds at any size (its columns sum to zero because every row of G sums
to zero).
"""
import os

import numpy as np
import pytest
import torch

import entropy_tcgen05_vocab_gb300 as flp
import workloads
from oracle import coracle, ref

pytestmark = pytest.mark.gpu
RTOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    flp.build()
    flp.lib()


def _rel(got, want, what):
    g = got.detach().cpu().double().numpy() if isinstance(got, torch.Tensor) else got
    assert np.all(np.isfinite(g)), what + ": non-finite"
    fro = np.linalg.norm(g - want) / max(np.linalg.norm(want), 1e-30)
    ele = np.abs(g - want).max() / max(np.abs(want).max(), 1e-30)
    assert fro <= RTOL and ele <= RTOL, "%s: rel Frobenius %.2e, rel max %.2e" % (what, fro, ele)
    return fro


def _case(T, H, V, dtype="bf16", seed=41, tau=0.7, all_rows=False):
    w = workloads.WORKLOADS[4].scaled(T=T, H=H, V=V, dtype=dtype, seed=seed, tau=tau)
    d = workloads.make(w, device="cuda")
    if all_rows:
        d["row_idx"] = None
        d["n"] = T
        g = torch.Generator().manual_seed(seed)
        d["g1"] = torch.randn(T, generator=g).cuda()
        d["g2"] = torch.randn(T, generator=g).cuda()
    return d


def _oracle(d, dtype):
    rows = None if d["row_idx"] is None else d["row_idx"].cpu().numpy()
    dh_rows, dW = coracle.backward(d["h"].cpu(), d["W"].cpu(), d["targets"].cpu().numpy(), rows,
                                   d["tau"], d["g1"].cpu().numpy(), d["g2"].cpu().numpy(), dtype)
    T = d["h"].shape[0]
    dh = coracle.scatter_rows(dh_rows, np.arange(T) if rows is None else rows, T)
    return dh, dW


@pytest.mark.parametrize("T,H,V,dtype", [
    (300, 256, 3000, "bf16"),     # several row/vocab tiles, ragged tails
    (260, 520, 3001, "bf16"),     # H not a multiple of 64 or 256; V odd (padded G rows)
    (200, 128, 2048, "fp16"),
    (129, 64, 300, "bf16"),
])
def test_backward_small(T, H, V, dtype):
    d = _case(T, H, V, dtype=dtype)
    dh, dW = flp.backward(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"], d["g1"], d["g2"])
    torch.cuda.synchronize()
    ref_dh, ref_dW = _oracle(d, dtype)
    _rel(dh, ref_dh, "dh")
    _rel(dW, ref_dW, "dW")
    scored = np.zeros(T, bool)
    scored[d["row_idx"].cpu().numpy()] = True
    assert torch.count_nonzero(dh[torch.from_numpy(~scored).cuda()]) == 0


def test_backward_all_rows_and_supplied_statistics():
    d = _case(384, 256, 4000, all_rows=True, tau=1.0)
    logp, ent, lse, ez = flp.logprob_entropy(d["h"], d["W"], d["targets"], None, 1.0,
                                             return_stats=True)
    a = flp.backward(d["h"], d["W"], d["targets"], None, 1.0, d["g1"], d["g2"])
    b = flp.backward(d["h"], d["W"], d["targets"], None, 1.0, d["g1"], d["g2"], lse, ez)
    torch.cuda.synchronize()
    ref_dh, ref_dW = _oracle(d, "bf16")
    for dh, dW in (a, b):
        _rel(dh, ref_dh, "dh")
        _rel(dW, ref_dW, "dW")


def test_backward_several_row_chunks(monkeypatch):
    d = _case(700, 256, 3000, seed=42)
    n = d["n"]
    monkeypatch.setenv("FLP_GRAD_CHUNK_ROWS", "128")
    assert len(flp.row_chunks(n, 128)) >= 3
    dh, dW = flp.backward(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"], d["g1"], d["g2"])
    torch.cuda.synchronize()
    ref_dh, ref_dW = _oracle(d, "bf16")
    _rel(dh, ref_dh, "dh")
    _rel(dW, ref_dW, "dW")


@pytest.mark.parametrize("T,H,V", [
    (600, 1024, 8192),    # 348 scored rows: 4 output tiles of dh, each in 8 K segments
    (2000, 512, 4100),    # 1205 rows: 5 tiles in K segments of 17, 17, 17, 14 k-blocks
])
def test_backward_dh_split_tail(monkeypatch, T, H, V):
    """When the dh GEMM's last wave of output tiles would leave most CTA
    pairs idle, those tiles are split along V into K segments whose FP32
    partials are added in a fixed order.  Against the oracle, against the
    unsplit GEMM (FLP_DH_SPLIT=0), and bitwise across repeated calls."""
    d = _case(T, H, V, seed=T + V)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    shape = flp.make_shape(T, H, V, d["n"], torch.bfloat16)
    pl = flp.plan(shape, flp.OP_BACKWARD, sms)
    assert pl["dh_split"] > 1 and pl["dh_tail_tiles"] > 0, pl
    args = (d["h"], d["W"], d["targets"], d["row_idx"], d["tau"], d["g1"], d["g2"])
    dh, dW = flp.backward(*args)
    dh2, _ = flp.backward(*args)
    monkeypatch.setenv("FLP_DH_SPLIT", "0")
    assert flp.plan(shape, flp.OP_BACKWARD, sms)["dh_split"] == 1
    dh_whole, dW_whole = flp.backward(*args)
    torch.cuda.synchronize()
    assert torch.equal(dh, dh2)
    assert torch.equal(dW, dW_whole)          # the dW GEMM does not change
    ref_dh, ref_dW = _oracle(d, "bf16")
    _rel(dh, ref_dh, "dh (split tail)")
    _rel(dh_whole, ref_dh, "dh (whole tiles)")
    _rel(dW, ref_dW, "dW")
    # the split changes only the FP32 summation order, so the two bf16
    # results differ by at most an ulp or so of the largest element
    diff = (dh.float() - dh_whole.float()).abs()
    assert diff.max().item() <= 2.0 ** -7 * dh_whole.float().abs().max().item()


@pytest.mark.parametrize("dtype,chunk", [("bf16", None), ("fp16", None), ("bf16", "128")])
def test_backward_repeated_rows_sum_their_contributions(monkeypatch, dtype, chunk):
    """row_idx naming rows 2, 3 and 5 times, scattered through the list (and,
    with 128-row chunks, across chunks): each such dh row is the sum of its
    contributions, as the oracle's scatter-add gives; dW takes every
    position."""
    d = _case(700, 256, 3000, dtype=dtype, seed=45)
    rows = d["row_idx"].cpu().numpy()
    extra = np.concatenate([rows[:5], rows[10:13], rows[10:13], np.repeat(rows[20:21], 4)])
    allrows = np.concatenate([rows, extra])[::-1].copy()
    allrows = np.roll(allrows, len(allrows) // 3)
    n = len(allrows)
    d["row_idx"] = torch.from_numpy(allrows).cuda()
    d["n"] = n
    d["g1"] = workloads.normal((n,), 1.0, 46, 1, "f32", "cpu").cuda()
    d["g2"] = workloads.normal((n,), 1.0, 46, 2, "f32", "cpu").cuda()
    if chunk:
        monkeypatch.setenv("FLP_GRAD_CHUNK_ROWS", chunk)
        assert len(flp.row_chunks(n, int(chunk))) >= 3
    dh, dW = flp.backward(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"], d["g1"], d["g2"])
    torch.cuda.synchronize()
    ref_dh, ref_dW = _oracle(d, dtype)
    _rel(dh, ref_dh, "dh")
    _rel(dW, ref_dW, "dW")
    # the repeated rows themselves, on their own
    rep = np.unique(extra)
    _rel(dh[torch.from_numpy(rep).cuda()], ref_dh[rep], "dh (repeated rows)")


def test_backward_frozen_weight_or_input_skips_that_gradient():
    """need_dW=False (a frozen output layer) or need_dh=False runs only the
    other GEMM; the gradient that is computed is bitwise the full call's."""
    d = _case(300, 256, 3000)
    args = (d["h"], d["W"], d["targets"], d["row_idx"], d["tau"], d["g1"], d["g2"])
    dh, dW = flp.backward(*args)
    dh_only, none_w = flp.backward(*args, need_dW=False)
    none_h, dW_only = flp.backward(*args, need_dh=False)
    assert none_w is None and none_h is None
    assert torch.equal(dh, dh_only) and torch.equal(dW, dW_only)
    with pytest.raises(ValueError):
        flp.backward(*args, need_dh=False, need_dW=False)


def test_autograd_with_a_frozen_weight():
    d = _case(300, 256, 3000)
    h = d["h"].clone().requires_grad_(True)
    logp, ent = flp.FusedLogProbEntropy.apply(h, d["W"], d["targets"], d["row_idx"], d["tau"])
    (logp * d["g1"] + ent * d["g2"]).sum().backward()
    dh, _ = flp.backward(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"], d["g1"], d["g2"])
    assert d["W"].grad is None
    assert torch.equal(h.grad, dh)


@pytest.mark.parametrize("tau", [0.1, 20.0])
def test_backward_extreme_temperatures(tau):
    d = _case(260, 128, 2500, seed=47, tau=tau)
    dh, dW = flp.backward(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"], d["g1"], d["g2"])
    torch.cuda.synchronize()
    ref_dh, ref_dW = _oracle(d, "bf16")
    _rel(dh, ref_dh, "dh")
    _rel(dW, ref_dW, "dW")


def test_backward_single_token_vocabulary_is_zero():
    """V = 1: p = 1 = the one-hot, z' = E z', so G and both gradients vanish."""
    d = _case(130, 64, 1, seed=48)
    dh, dW = flp.backward(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"], d["g1"], d["g2"])
    assert dh.float().abs().max().item() <= 1e-5 and dW.abs().max().item() <= 1e-5


def test_backward_no_scored_rows_gives_zeros():
    d = _case(64, 128, 512)
    rows = torch.zeros(0, dtype=torch.int64, device="cuda")
    e = torch.zeros(0, device="cuda")
    dh, dW = flp.backward(d["h"], d["W"], d["targets"], rows, 0.7, e, e)
    assert torch.count_nonzero(dh) == 0 and torch.count_nonzero(dW) == 0


def test_autograd_function_matches_backward():
    d = _case(256, 128, 2000, seed=43)
    h = d["h"].clone().requires_grad_(True)
    W = d["W"].clone().requires_grad_(True)
    logp, ent = flp.FusedLogProbEntropy.apply(h, W, d["targets"], d["row_idx"], d["tau"])
    (logp * d["g1"] + ent * d["g2"]).sum().backward()
    dh, dW = flp.backward(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"], d["g1"], d["g2"])
    assert torch.equal(h.grad, dh)
    assert torch.allclose(W.grad.float(), dW.to(torch.bfloat16).float())


def test_backward_workload_full_size():
    d = workloads.make(4, device="cuda")
    dh, dW = flp.backward(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"], d["g1"], d["g2"])
    logp, _, lse, ez = flp.logprob_entropy(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"],
                                           return_stats=True)
    torch.cuda.synchronize()
    n = d["n"]
    rows = d["row_idx"].cpu().numpy()
    tg = d["targets"].cpu().numpy()
    # every scored row's statistics in float64 (dW[v] sums over all of them);
    # the kernels' own statistics are checked against them on the way
    hd, Wd = ref.decode(d["h"].cpu(), "bf16"), ref.decode(d["W"].cpu(), "bf16")
    lse_ref, ez_ref = ref.row_stats(hd, Wd, rows, d["tau"])
    del hd, Wd
    assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= 1e-3
    assert np.abs(ez.cpu().double().numpy() - ez_ref).max() <= 1e-3
    # dh on 512 sampled scored rows and the 8 with the most negative log-prob;
    # dW on 256 sampled vocabulary rows, those rows' targets and the last row
    worst = np.argsort(logp.cpu().numpy())[:8]
    sel = np.unique(np.concatenate([workloads.sample_rows(n, 512, seed=4), worst]))
    vsel = np.unique(np.concatenate([workloads.sample_rows(d["workload"].V, 256, seed=44),
                                     tg[rows[worst]], [d["workload"].V - 1]]))
    want_dh, want_dW = ref.backward(d["h"].cpu(), d["W"].cpu(), tg, rows, d["tau"],
                                    d["g1"].cpu().numpy(), d["g2"].cpu().numpy(), "bf16",
                                    dh_rows_sel=sel, vsel=vsel, stats=(lse_ref, ez_ref))
    _rel(dh[torch.from_numpy(rows[sel]).cuda()], want_dh, "dh (sampled rows)")
    _rel(dW[torch.from_numpy(vsel).cuda()], want_dW, "dW (sampled vocabulary rows)")
    # unscored rows are zero
    scored = torch.zeros(d["h"].shape[0], dtype=torch.bool, device="cuda")
    scored[d["row_idx"]] = True
    assert torch.count_nonzero(dh[~scored]) == 0
    # dW: every row of G sums to zero, so the columns of dW sum to zero
    colsum = dW.double().sum(0)
    scale = dW.double().abs().sum(0)
    assert torch.all(colsum.abs() <= 2e-3 * scale), (colsum.abs() / scale).max()
    assert torch.isfinite(dW).all()


def test_backward_dw_rows_exact_at_full_vocabulary():
    # same H, V and launch shape as the full workload, 1,200 scored rows
    w = workloads.WORKLOADS[4].scaled(T=2000)
    d = workloads.make(w, device="cuda")
    rows = d["row_idx"].cpu().numpy()
    dh, dW = flp.backward(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"], d["g1"], d["g2"])
    torch.cuda.synchronize()
    vsel = np.concatenate([workloads.sample_rows(w.V, 256, seed=44),
                           d["targets"].cpu().numpy()[rows[:8]], [w.V - 1]])
    _, want = ref.backward(d["h"].cpu(), d["W"].cpu(), d["targets"].cpu().numpy(), rows, d["tau"],
                           d["g1"].cpu().numpy(), d["g2"].cpu().numpy(), "bf16",
                           dh_rows_sel=np.zeros(0, np.int64), vsel=vsel)
    _rel(dW[torch.from_numpy(vsel).cuda()], want, "dW (sampled vocabulary rows)")


def test_backward_repeated_calls_are_bitwise_identical():
    d = _case(300, 256, 3000)
    a = flp.backward(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"], d["g1"], d["g2"])
    b = flp.backward(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"], d["g1"], d["g2"])
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
