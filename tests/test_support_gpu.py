"""GPU parity of the sampling-support entry points against the float64 oracle.

flp_logprob_entropy_support / flp_backward_support restrict each row's
softmax to its sampling support (a bitmask of uint32 words by h row) and
flp_pack_support builds that bitmask from a byte-per-token mask.  Compared
element by element with the oracle on small cases that span several row
tiles, vocabulary tiles and splits with ragged tails, at several support
densities; on sampled rows at the full forward-scoring size (4096 x 4096 x
151,936, tau 0.7) with a 1/32-dense support.  Edge cases: every token kept
(equals the unrestricted kernel), padded rows of words with garbage past V,
a target outside the support (-inf), an empty support (NaN, counted), a
support that leaves out each row's dominant logit, a support inside one
vocabulary tile.  Tolerances: |d logp|, |d ent| <= 1e-3; gradients 1e-2
relative (Frobenius and max element).
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
RTOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    flp.build()
    flp.lib()


def _check(got, want, what, tol=TOL):
    got = got.detach().cpu().double().numpy()
    fin = np.isfinite(want)
    assert np.array_equal(np.isfinite(got), fin), what + ": finite pattern differs"
    assert np.array_equal(got[~fin], want[~fin]) or np.array_equal(
        np.isnan(got[~fin]), np.isnan(want[~fin])), what + ": non-finite values differ"
    if fin.any():
        err = np.abs(got[fin] - want[fin])
        assert err.max() <= tol, "%s: max |diff| %.3e" % (what, err.max())


def _case(T, H, V, j, seed, dtype="bf16", rows=False, ld=None):
    w = workloads.WORKLOADS[0].scaled(T=T, H=H, V=V, seed=seed, w_std=0.08, dtype=dtype)
    d = workloads.make(w, device="cuda")
    sup = workloads.support_words(T, V, j, seed, targets=d["targets"].cpu().numpy(), ld=ld)
    d["support"] = torch.from_numpy(sup).cuda()
    d["sup_np"] = sup
    d["rows"] = None
    if rows:
        d["rows"] = torch.from_numpy(workloads.sample_rows(T, T // 2, seed=seed)).cuda()
    return d


def _compare(d, tau, dt="bf16"):
    logp, ent, lse, ez = flp.logprob_entropy(d["h"], d["W"], d["targets"], d["rows"], tau,
                                             return_stats=True, support=d["support"])
    torch.cuda.synchronize()
    rows = None if d["rows"] is None else d["rows"].cpu().numpy()
    o = coracle.logprob_entropy_support(d["h"].cpu(), d["W"].cpu(), d["targets"].cpu().numpy(),
                                        rows, d["sup_np"], tau, dt)
    _check(logp, o["logp"], "logp")
    _check(ent, o["ent"], "ent")
    _check(lse, o["lse"], "lse")
    _check(ez, o["ez"], "ez", tol=2e-3)
    return logp, ent


@pytest.mark.parametrize("T,H,V,j,rows", [
    (300, 256, 5000, 1, False),    # half the tokens, several row and vocabulary tiles
    (260, 192, 8200, 3, True),     # 1/8 of the tokens, row subset, last vocab tile 8 columns
    (129, 64, 1000, 6, False),     # ~15 tokens per row
    (40, 96, 33, 1, False),        # V one past a 32-column chunk
    (1000, 128, 20000, 5, True),   # many tiles and splits, 1/32 of the tokens
])
def test_support_small(T, H, V, j, rows):
    _compare(_case(T, H, V, j, seed=T + V + j, rows=rows), 0.7)


@pytest.mark.parametrize("n", [100, 128, 129])
def test_support_both_sides_of_the_few_rows_switch(n):
    """n <= 128 scored rows run the single-CTA kernel, more the CTA pairs."""
    d = _case(400, 256, 33000, 4, seed=n + 7)
    d["rows"] = torch.from_numpy(workloads.sample_rows(400, n, seed=n)).cuda()
    _compare(d, 0.7)


def test_support_fp16():
    _compare(_case(200, 256, 6000, 2, seed=61, dtype="fp16"), 1.0, dt="fp16")


def test_every_token_kept_equals_the_unrestricted_kernel():
    d = _case(300, 256, 5000, 0, seed=62)
    a = flp.logprob_entropy(d["h"], d["W"], d["targets"], None, 0.8, support=d["support"])
    b = flp.logprob_entropy(d["h"], d["W"], d["targets"], None, 0.8)
    for x, y in zip(a, b):
        assert torch.allclose(x, y, rtol=0, atol=1e-5)


def test_padded_words_and_bits_past_v_are_ignored():
    d = _case(150, 128, 1000, 1, seed=63, ld=40)           # 32 words used, 8 of padding
    words = d["sup_np"].view(np.uint32).copy()
    clean = words.copy()
    clean[:, 31] &= np.uint32((1 << (1000 - 31 * 32)) - 1)  # only bits < V
    clean[:, 32:] = 0
    a = flp.logprob_entropy(d["h"], d["W"], d["targets"], None, 1.0, support=d["support"])
    b = flp.logprob_entropy(d["h"], d["W"], d["targets"], None, 1.0,
                            support=torch.from_numpy(clean.view(np.int32)).cuda())
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    _compare(d, 1.0)


def test_target_off_support_and_empty_support():
    d = _case(300, 128, 3000, 2, seed=64)
    words = d["sup_np"].view(np.uint32).copy()
    tg = d["targets"].cpu().numpy()
    for r in (3, 200):
        words[r, tg[r] // 32] &= ~np.uint32(1 << (tg[r] % 32))
    words[7] = 0
    words[299] = 0
    d["sup_np"] = words.view(np.int32)
    d["support"] = torch.from_numpy(d["sup_np"]).cuda()
    shape = flp.make_shape(300, 128, 3000, 300, torch.bfloat16)
    ws = torch.empty(flp.workspace_size(shape, flp.OP_LOGPROB_ENTROPY), dtype=torch.uint8,
                     device="cuda")
    logp, ent = flp.logprob_entropy(d["h"], d["W"], d["targets"], None, 0.9, workspace=ws,
                                    support=d["support"])
    st = flp.read_device_status(ws)
    assert st == {"bad_targets": 0, "bad_rows": 0, "timeouts": 0, "empty_supports": 2}
    lp, en = logp.cpu().numpy(), ent.cpu().numpy()
    assert lp[3] == -np.inf and lp[200] == -np.inf and np.isfinite(en[[3, 200]]).all()
    assert np.isnan(lp[[7, 299]]).all() and np.isnan(en[[7, 299]]).all()
    _compare(d, 0.9)


def test_support_without_the_dominant_logit():
    """Each checked row has one logit ~70 above the rest; the support leaves it
    out, so the support's maximum is far below the row's maximum."""
    g = torch.Generator().manual_seed(65)
    T, H, V = 260, 64, 3000
    h = torch.randn(T, H, generator=g, dtype=torch.float64)
    W = torch.randn(V, H, generator=g, dtype=torch.float64) * 0.01
    dom = torch.randperm(V, generator=g)[:T]
    for i in range(0, T, 13):
        W[dom[i]] = 70.0 * h[i] / (h[i] @ h[i])
    hb, Wb = h.to(torch.bfloat16), W.to(torch.bfloat16)
    tg = torch.randint(0, V, (T,), generator=g).numpy()
    sup = workloads.support_words(T, V, 1, 65, targets=tg).view(np.uint32)
    for i in range(T):
        sup[i, int(dom[i]) // 32] &= ~np.uint32(1 << (int(dom[i]) % 32))
        sup[i, tg[i] // 32] |= np.uint32(1 << (tg[i] % 32))
    d = {"h": hb.cuda(), "W": Wb.cuda(), "targets": torch.from_numpy(tg).cuda(),
         "rows": torch.arange(0, T, 13).cuda(), "sup_np": sup.view(np.int32)}
    d["support"] = torch.from_numpy(d["sup_np"]).cuda()
    _compare(d, 1.0)


def test_support_inside_one_vocabulary_tile():
    d = _case(300, 128, 30000, 0, seed=66)
    words = np.zeros_like(d["sup_np"].view(np.uint32))
    words[:, 18:22] = 0xFFFFFFFF                           # tokens 576 .. 703
    tg = 600 + (np.arange(300) * 7) % 100
    d["targets"] = torch.from_numpy(tg).cuda()
    d["sup_np"] = words.view(np.int32)
    d["support"] = torch.from_numpy(d["sup_np"]).cuda()
    _compare(d, 0.7)


@pytest.mark.parametrize("T,V,ld_mask", [(5, 70, 70), (300, 1000, 1024), (33, 32, 40)])
def test_pack_support(T, V, ld_mask):
    g = torch.Generator().manual_seed(T + V)
    full = torch.rand(T, ld_mask, generator=g) < 0.4
    mask = full.cuda()[:, :V]
    words = flp.pack_support(mask)
    want = np.packbits(full[:, :V].numpy(), axis=1, bitorder="little")
    want = np.pad(want, ((0, 0), (0, 4 * ((V + 31) // 32) - want.shape[1])))
    assert torch.equal(words.cpu(), torch.from_numpy(want.view(np.int32)))
    padded = flp.pack_support(mask.to(torch.uint8), words=(V + 31) // 32 + 3)
    assert torch.equal(padded[:, :words.shape[1]].cpu(), words.cpu())
    assert torch.count_nonzero(padded[:, words.shape[1]:]) == 0


def test_forward_scoring_workload_with_support_sampled():
    d = workloads.make(1, device="cuda")
    tg = d["targets"].cpu().numpy()
    sup = workloads.support_words(4096, d["workload"].V, 5, 1, targets=tg)
    logp, ent = flp.logprob_entropy(d["h"], d["W"], d["targets"], None, d["tau"],
                                    support=torch.from_numpy(sup).cuda())
    torch.cuda.synchronize()
    pos = np.unique(np.concatenate([workloads.sample_rows(4096, 192, seed=67), [0, 4095]]))
    o = ref.logprob_entropy(d["h"].cpu(), d["W"].cpu(), tg, pos, d["tau"], "bf16", support=sup)
    _check(logp[torch.from_numpy(pos).cuda()], o["logp"], "logp")
    _check(ent[torch.from_numpy(pos).cuda()], o["ent"], "ent")
    lp, en = logp.cpu().numpy(), ent.cpu().numpy()
    assert np.all(np.isfinite(lp)) and np.all(lp <= 1e-4)
    assert np.all(en >= -1e-4) and np.all(en <= math.log(d["workload"].V / 16))


# ---------------------------------------------------------------- backward

def _rel(got, want, what):
    g = got.detach().cpu().double().numpy()
    assert np.all(np.isfinite(g)), what + ": non-finite"
    fro = np.linalg.norm(g - want) / max(np.linalg.norm(want), 1e-30)
    ele = np.abs(g - want).max() / max(np.abs(want).max(), 1e-30)
    assert fro <= RTOL and ele <= RTOL, "%s: rel Frobenius %.2e, rel max %.2e" % (what, fro, ele)


@pytest.mark.parametrize("T,H,V,j", [(300, 256, 3000, 1), (260, 136, 3001, 3), (129, 64, 600, 5)])
def test_support_backward(T, H, V, j):
    w = workloads.WORKLOADS[4].scaled(T=T, H=H, V=V, seed=T + j, tau=0.7)
    d = workloads.make(w, device="cuda")
    tg = d["targets"].cpu().numpy()
    words = workloads.support_words(T, V, j, T + j, targets=tg).view(np.uint32)
    rows = d["row_idx"].cpu().numpy()
    r_off = rows[1]                                           # one target outside its support
    words[r_off, tg[r_off] // 32] &= ~np.uint32(1 << (tg[r_off] % 32))
    sup = words.view(np.int32)
    support = torch.from_numpy(sup).cuda()
    dh, dW = flp.backward(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"], d["g1"], d["g2"],
                          support=support)
    torch.cuda.synchronize()
    dh_rows, ref_dW = coracle.backward_support(d["h"].cpu(), d["W"].cpu(), tg, rows, sup, d["tau"],
                                               d["g1"].cpu().numpy(), d["g2"].cpu().numpy(),
                                               "bf16")
    _rel(dh, coracle.scatter_rows(dh_rows, rows, T), "dh")
    _rel(dW, ref_dW, "dW")
    # tokens outside every scored row's support get exactly zero gradient
    keep = ref.support_bits(sup, rows, V).any(axis=0)
    if (~keep).any():
        assert torch.count_nonzero(dW[torch.from_numpy(~keep).cuda()]) == 0
    # statistics from the forward give the same result as recomputing them
    _, _, lse, ez = flp.logprob_entropy(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"],
                                        return_stats=True, support=support)
    dh2, dW2 = flp.backward(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"], d["g1"],
                            d["g2"], lse, ez, support=support)
    assert torch.allclose(dh2.float(), dh.float(), rtol=0, atol=1e-3 * dh.float().abs().max())
    assert torch.allclose(dW2, dW, rtol=0, atol=1e-3 * dW.abs().max())


def test_autograd_with_support():
    w = workloads.WORKLOADS[4].scaled(T=200, H=128, V=2000, seed=68, tau=0.9)
    d = workloads.make(w, device="cuda")
    support = torch.from_numpy(workloads.support_words(200, 2000, 2, 68,
                                                       targets=d["targets"].cpu().numpy())).cuda()
    h = d["h"].clone().requires_grad_(True)
    W = d["W"].clone().requires_grad_(True)
    logp, ent = flp.FusedLogProbEntropy.apply(h, W, d["targets"], d["row_idx"], 0.9, support)
    (d["g1"] * logp + d["g2"] * ent).sum().backward()
    dh, dW = flp.backward(d["h"], d["W"], d["targets"], d["row_idx"], 0.9, d["g1"], d["g2"],
                          support=support)
    assert torch.allclose(h.grad.float(), dh.float(), rtol=0, atol=1e-3 * dh.float().abs().max())
    assert torch.allclose(W.grad.float(), dW.to(W.dtype).float(), rtol=0,
                          atol=1e-2 * dW.abs().max())


def test_support_repeated_calls_are_bitwise_identical():
    d = _case(300, 256, 5000, 2, seed=83)
    a = flp.logprob_entropy(d["h"], d["W"], d["targets"], None, 0.7, support=d["support"])
    b = flp.logprob_entropy(d["h"], d["W"], d["targets"], None, 0.7, support=d["support"])
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_support_backward_full_backward_workload():
    """The backward workload (16,384 rows, 60 % scored, H 4096, V 151,936,
    tau 0.7) restricted to 1/32-dense supports: dh on sampled scored rows
    against the oracle, unscored rows zero, and the columns of dW summing to
    zero (each row of G sums to zero over its support)."""
    d = workloads.make(4, device="cuda")
    w = d["workload"]
    tg = d["targets"].cpu().numpy()
    sup = workloads.support_words(w.T, w.V, 5, 4, targets=tg)
    dh, dW = flp.backward(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"], d["g1"], d["g2"],
                          support=torch.from_numpy(sup).cuda())
    torch.cuda.synchronize()
    n = d["n"]
    rows = d["row_idx"].cpu().numpy()
    sel = workloads.sample_rows(n, 64, seed=84)
    want, _ = ref.backward(d["h"].cpu(), d["W"].cpu(), tg, rows, d["tau"], d["g1"].cpu().numpy(),
                           d["g2"].cpu().numpy(), "bf16", dh_rows_sel=sel,
                           vsel=np.zeros(0, np.int64), stats=(np.zeros(n), np.zeros(n)),
                           support=sup)
    _rel(dh[torch.from_numpy(rows[sel]).cuda()], want, "dh (sampled rows)")
    scored = torch.zeros(w.T, dtype=torch.bool, device="cuda")
    scored[d["row_idx"]] = True
    assert torch.count_nonzero(dh[~scored]) == 0
    colsum = dW.double().sum(0)
    scale = dW.double().abs().sum(0)
    assert torch.all(colsum.abs() <= 2e-3 * scale), (colsum.abs() / scale).max()
    assert torch.isfinite(dW).all()
