"""Pins for the float64 oracle (CPU only).

The oracle is the reference every GPU parity test trusts, so it is pinned
here to things other than itself: exact decoding of every storage bit
pattern, closed forms (W = 0, one dominant logit, two classes, identical
KL heads), invariants (shift, temperature as a scale, row subsets and
order), 50-digit brute force on tiny inputs, and central finite
differences of its own forward for the backward.  Each C-oracle result is
also cross-checked against the independent NumPy restatement.
"""
import math
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

from oracle import coracle, ref
import workloads

LN = math.log


def _bits(x, dtype):
    t = torch.as_tensor(x, dtype=torch.float32).to(workloads.TORCH_DTYPES[dtype])
    return t.view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------
# storage decoding

def test_decode_every_bf16_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    for got in (coracle.decode(bits, "bf16"), ref.decode(bits, "bf16")):
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan], want[~nan])


def test_decode_every_fp16_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.float16).double().numpy()
    for got in (coracle.decode(bits, "fp16"), ref.decode(bits, "fp16")):
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan], want[~nan])
    # spot values of the format itself
    assert coracle.decode(np.array([0x3C00, 0x0001, 0x7BFF, 0xC000], np.uint16), "fp16").tolist() \
        == [1.0, 2.0 ** -24, 65504.0, -2.0]


# --------------------------------------------------------------------------
# closed forms

@pytest.mark.parametrize("V,H", [(8192, 16), (151936, 8), (38016, 8)])
@pytest.mark.parametrize("tau", [0.7, 1.0, 3.0])
def test_zero_weight_gives_uniform(V, H, tau):
    rng = np.random.default_rng(0)
    h = _bits(rng.standard_normal((3, H)), "bf16")
    W = np.zeros((V, H), np.uint16)                      # +0.0 in bf16
    tg = rng.integers(0, V, size=3)
    o = coracle.logprob_entropy(h, W, tg, None, tau, "bf16")
    np.testing.assert_allclose(o["logp"], -LN(V), rtol=0, atol=1e-12)
    np.testing.assert_allclose(o["ent"], LN(V), rtol=0, atol=1e-12)
    if V == 8192:
        assert abs(LN(V) - 9.010913) < 1e-6
    if V == 151936:
        assert abs(LN(V) - 11.931215) < 1e-6


def test_one_hot_dominant_row():
    """W[tgt] = c h / |h|^2 puts logit c on the target; the rest are O(1)."""
    rng = np.random.default_rng(1)
    H, V = 64, 1000
    hf = rng.standard_normal((4, H))
    Wf = rng.standard_normal((V, H)) * 0.01
    tg = np.array([3, 500, 999, 0])
    for i in range(4):
        Wf[tg[i]] = 60.0 * hf[i] / (hf[i] @ hf[i])
    o = coracle.logprob_entropy(hf, Wf, tg, None, 1.0, "f64")
    z = hf @ Wf.T
    for i in range(4):
        margin = z[i, tg[i]] - np.max(np.delete(z[i], tg[i]))
        assert margin >= 40
    assert np.all(o["logp"] <= 0) and np.all(o["logp"] >= -V * math.exp(-40))
    assert np.all(o["ent"] >= 0) and np.all(o["ent"] <= V * math.exp(-40) * 62)


@pytest.mark.parametrize("tau", [0.5, 1.0, 2.0])
def test_two_classes(tau):
    rng = np.random.default_rng(2)
    h = rng.standard_normal((5, 3))
    W = rng.standard_normal((2, 3))
    tg = np.array([0, 1, 1, 0, 1])
    o = coracle.logprob_entropy(h, W, tg, None, tau, "f64")
    z = h @ W.T / tau
    for i in range(5):
        d = z[i, tg[i]] - z[i, 1 - tg[i]]
        assert o["logp"][i] == pytest.approx(-math.log1p(math.exp(-d)), abs=1e-13)
        p = 1.0 / (1.0 + math.exp(-(z[i, 0] - z[i, 1])))
        assert o["ent"][i] == pytest.approx(-(p * LN(p) + (1 - p) * LN(1 - p)), abs=1e-13)


def test_large_temperature_entropy_tends_to_log_v():
    rng = np.random.default_rng(3)
    h = rng.standard_normal((2, 16))
    W = rng.standard_normal((100, 16))
    tg = np.array([1, 2])
    o = coracle.logprob_entropy(h, W, tg, None, 1e6, "f64")
    np.testing.assert_allclose(o["ent"], LN(100), atol=1e-8)
    np.testing.assert_allclose(o["logp"], -LN(100), atol=1e-4)


# --------------------------------------------------------------------------
# invariants

def _random_case(seed, T=12, H=24, V=300, dtype="bf16"):
    w = workloads.WORKLOADS[0].scaled(T=T, H=H, V=V, dtype=dtype, seed=seed, w_std=0.3)
    return workloads.make(w)


def test_bounds_on_config0():
    d = workloads.make(0)
    o = coracle.logprob_entropy(d["h"], d["W"], d["targets"], None, 1.0, "bf16")
    assert o["rc"] == 0
    assert np.all(o["logp"] <= 0)
    assert np.all(o["ent"] >= 0) and np.all(o["ent"] <= LN(8192))


def test_shift_invariance():
    """Append a column: every logit of a row shifts by s_r c; outputs do not move."""
    rng = np.random.default_rng(4)
    h = rng.standard_normal((6, 10))
    W = rng.standard_normal((50, 10)) * 0.5
    tg = rng.integers(0, 50, size=6)
    s = rng.standard_normal((6, 1)) * 3
    h2 = np.hstack([h, s])
    W2 = np.hstack([W, np.full((50, 1), 2.5)])
    for tau in (0.7, 1.0):
        a = coracle.logprob_entropy(h, W, tg, None, tau, "f64")
        b = coracle.logprob_entropy(h2, W2, tg, None, tau, "f64")
        for k in ("logp", "ent", "ez"):
            if k == "ez":
                np.testing.assert_allclose(b[k] - a[k], (s[:, 0] * 2.5) / tau, atol=1e-10)
            else:
                np.testing.assert_allclose(a[k], b[k], atol=1e-11)


def test_temperature_is_a_scale_of_the_logits():
    rng = np.random.default_rng(5)
    h = rng.standard_normal((7, 9))
    W = rng.standard_normal((40, 9))
    tg = rng.integers(0, 40, size=7)
    a = coracle.logprob_entropy(h, W, tg, None, 0.7, "f64")
    b = coracle.logprob_entropy(h, W / 0.7, tg, None, 1.0, "f64")
    for k in ("logp", "ent", "lse", "ez"):
        np.testing.assert_allclose(a[k], b[k], rtol=1e-12, atol=1e-12)


def test_row_subsets_and_order_do_not_matter():
    """Chunked equals unchunked: any split, order or repetition of rows."""
    d = _random_case(6, T=40)
    full = coracle.logprob_entropy(d["h"], d["W"], d["targets"], None, 0.7, "bf16")
    rows = np.array([39, 0, 5, 5, 17, 38, 1])
    part = coracle.logprob_entropy(d["h"], d["W"], d["targets"], rows, 0.7, "bf16")
    for k in ("logp", "ent", "lse", "ez"):
        np.testing.assert_array_equal(part[k], full[k][rows])
    for chunk in (1, 3, 16):
        got = np.concatenate([
            coracle.logprob_entropy(d["h"], d["W"], d["targets"], np.arange(i, min(i + chunk, 40)),
                                    0.7, "bf16")["logp"] for i in range(0, 40, chunk)])
        np.testing.assert_array_equal(got, full["logp"])


def test_targets_follow_the_original_row():
    d = _random_case(7, T=10)
    rows = np.array([9, 2, 4])
    tg = d["targets"].numpy().copy()
    o = coracle.logprob_entropy(d["h"], d["W"], tg, rows, 1.0, "bf16")
    hd = ref.decode(d["h"], "bf16")
    Wd = ref.decode(d["W"], "bf16")
    for i, r in enumerate(rows):
        z = hd[r] @ Wd.T
        m = z.max()
        lse = m + LN(np.exp(z - m).sum())
        assert o["logp"][i] == pytest.approx(z[tg[r]] - lse, abs=1e-12)


def test_bad_target_and_row_give_nan():
    d = _random_case(8, T=6)
    tg = d["targets"].numpy().copy()
    tg[2] = 10 ** 6
    o = coracle.logprob_entropy(d["h"], d["W"], tg, np.array([0, 2, 7, 1]), 1.0, "bf16")
    assert o["rc"] == -1
    assert np.isnan(o["logp"][1]) and np.isfinite(o["ent"][1])
    assert np.isnan(o["logp"][2]) and np.isnan(o["ent"][2])
    assert np.isfinite(o["logp"][0]) and np.isfinite(o["logp"][3])


# --------------------------------------------------------------------------
# 50-digit brute force on tiny inputs

def _dec_forward(h, W, tg, rows, tau):
    getcontext().prec = 50
    out = []
    for r in rows:
        z = [sum(Decimal(float(h[r, k])) * Decimal(float(W[v, k])) for k in range(h.shape[1]))
             / Decimal(repr(tau)) for v in range(W.shape[0])]
        S = sum((x.exp() for x in z), Decimal(0))
        lse = S.ln()
        ez = sum(((x - lse).exp() * x for x in z), Decimal(0))
        out.append((float(z[tg[r]] - lse), float(lse - ez), float(lse), float(ez)))
    return np.array(out)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("tau", [0.7, 1.0])
def test_brute_force_forward(dtype, tau):
    d = _random_case(9, T=7, H=13, V=37, dtype=dtype)
    rows = np.array([6, 0, 3, 3])
    tg = d["targets"].numpy()
    hd, Wd = ref.decode(d["h"], dtype), ref.decode(d["W"], dtype)
    want = _dec_forward(hd, Wd, tg, rows, tau)
    c = coracle.logprob_entropy(d["h"], d["W"], tg, rows, tau, dtype)
    n = ref.logprob_entropy(d["h"], d["W"], tg, rows, tau, dtype)
    for o in (c, n):
        got = np.stack([o["logp"], o["ent"], o["lse"], o["ez"]], axis=1)
        np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)


def _dec_kl(hs, Ws, ht, Wt, rows):
    getcontext().prec = 50
    out = []
    for r in rows:
        def lsm(h, W):
            z = [sum(Decimal(float(h[r, k])) * Decimal(float(W[v, k])) for k in range(h.shape[1]))
                 for v in range(W.shape[0])]
            L = sum((x.exp() for x in z), Decimal(0)).ln()
            return [x - L for x in z]
        ls, lt = lsm(hs, Ws), lsm(ht, Wt)
        out.append(float(sum((b.exp() * (b - a) for a, b in zip(ls, lt)), Decimal(0))))
    return np.array(out)


def test_brute_force_kl():
    w = workloads.WORKLOADS[3].scaled(T=5, H=11, V=29, w_std=0.4, seed=10)
    d = workloads.make(w)
    rows = np.array([4, 1, 0])
    dec = [ref.decode(d[k], "bf16") for k in ("h_s", "W_s", "h_t", "W_t")]
    want = _dec_kl(*dec, rows)
    np.testing.assert_allclose(coracle.kl(d["h_s"], d["W_s"], d["h_t"], d["W_t"], rows, "bf16"),
                               want, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(ref.kl(d["h_s"], d["W_s"], d["h_t"], d["W_t"], rows, "bf16"),
                               want, rtol=1e-12, atol=1e-14)


def test_kl_closed_forms():
    w = workloads.WORKLOADS[3].scaled(T=6, H=16, V=64, seed=11)
    d = workloads.make(w)
    same = coracle.kl(d["h_s"], d["W_s"], d["h_s"], d["W_s"], None, "bf16")
    assert np.all(np.abs(same) < 1e-14)
    diff = coracle.kl(d["h_s"], d["W_s"], d["h_t"], d["W_t"], None, "bf16")
    assert np.all(diff > 0)
    # two classes: KL of Bernoulli(q) from Bernoulli(p)
    rng = np.random.default_rng(12)
    hs, ht = rng.standard_normal((3, 4)), rng.standard_normal((3, 4))
    Ws, Wt = rng.standard_normal((2, 4)), rng.standard_normal((2, 4))
    got = coracle.kl(hs, Ws, ht, Wt, None, "f64")
    for i in range(3):
        zs, zt = hs[i] @ Ws.T, ht[i] @ Wt.T
        p = 1 / (1 + math.exp(zs[1] - zs[0]))
        q = 1 / (1 + math.exp(zt[1] - zt[0]))
        assert got[i] == pytest.approx(q * LN(q / p) + (1 - q) * LN((1 - q) / (1 - p)), abs=1e-13)


# --------------------------------------------------------------------------
# backward

def _loss(h, W, tg, rows, tau, g1, g2):
    o = coracle.logprob_entropy(h, W, tg, rows, tau, "f64")
    return float(np.sum(g1 * o["logp"] + g2 * o["ent"]))


@pytest.mark.parametrize("tau,rows", [
    (0.7, [5, 0, 2, 3]),
    (1.0, [5, 0, 2, 3]),
    (0.7, [5, 0, 2, 5, 3, 0, 5]),   # rows scored more than once: their terms add up
])
def test_backward_matches_finite_differences(tau, rows):
    rng = np.random.default_rng(13)
    T, H, V = 6, 5, 7
    h = rng.standard_normal((T, H))
    W = rng.standard_normal((V, H)) * 0.7
    tg = rng.integers(0, V, size=T)
    rows = np.array(rows)
    g1, g2 = rng.standard_normal(len(rows)), rng.standard_normal(len(rows))
    dh_rows, dW = coracle.backward(h, W, tg, rows, tau, g1, g2, "f64")
    dh = coracle.scatter_rows(dh_rows, rows, T)
    eps = 1e-6
    num_h = np.zeros_like(h)
    for r in range(T):
        for k in range(H):
            hp, hm = h.copy(), h.copy()
            hp[r, k] += eps
            hm[r, k] -= eps
            num_h[r, k] = (_loss(hp, W, tg, rows, tau, g1, g2)
                           - _loss(hm, W, tg, rows, tau, g1, g2)) / (2 * eps)
    num_W = np.zeros_like(W)
    for v in range(V):
        for k in range(H):
            Wp, Wm = W.copy(), W.copy()
            Wp[v, k] += eps
            Wm[v, k] -= eps
            num_W[v, k] = (_loss(h, Wp, tg, rows, tau, g1, g2)
                           - _loss(h, Wm, tg, rows, tau, g1, g2)) / (2 * eps)
    assert np.linalg.norm(dh - num_h) <= 1e-6 * np.linalg.norm(num_h)
    assert np.linalg.norm(dW - num_W) <= 1e-6 * np.linalg.norm(num_W)
    assert np.all(dh[[1, 4]] == 0)                     # unscored rows
    rdh, rdW = ref.backward(h, W, tg, rows, tau, g1, g2, "f64")
    np.testing.assert_allclose(rdh, dh_rows, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(rdW, dW, rtol=1e-10, atol=1e-12)


def test_backward_dw_columns_sum_to_zero():
    """sum_v G_rv = 0 for every row, hence sum_v dW[v,:] = 0."""
    w = workloads.WORKLOADS[4].scaled(T=24, H=32, V=500, seed=14)
    d = workloads.make(w)
    rows = d["row_idx"].numpy()
    _, dW = coracle.backward(d["h"], d["W"], d["targets"], rows, 0.7, d["g1"].numpy(),
                             d["g2"].numpy(), "bf16", want_dh=False)
    scale = np.abs(dW).sum(axis=0)
    assert np.all(np.abs(dW.sum(axis=0)) <= 1e-12 * scale + 1e-15)


def test_backward_subsets_match_full():
    w = workloads.WORKLOADS[4].scaled(T=30, H=24, V=260, seed=15)
    d = workloads.make(w)
    rows = d["row_idx"].numpy()
    g1, g2 = d["g1"].numpy(), d["g2"].numpy()
    dh, dW = coracle.backward(d["h"], d["W"], d["targets"], rows, 0.7, g1, g2, "bf16")
    vsel = np.array([0, 7, 259, 100])
    _, dWs = coracle.backward(d["h"], d["W"], d["targets"], rows, 0.7, g1, g2, "bf16",
                              want_dh=False, vsel=vsel)
    np.testing.assert_allclose(dWs, dW[vsel], rtol=1e-13, atol=1e-15)
    sel = np.array([2, 0])
    rdh, rdW = ref.backward(d["h"], d["W"], d["targets"], rows, 0.7, g1, g2, "bf16",
                            dh_rows_sel=sel, vsel=vsel)
    np.testing.assert_allclose(rdh, dh[sel], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(rdW, dW[vsel], rtol=1e-10, atol=1e-13)


# --------------------------------------------------------------------------
# the two restatements agree on real workload shapes

def test_c_and_numpy_agree_config0():
    d = workloads.make(0)
    c = coracle.logprob_entropy(d["h"], d["W"], d["targets"], None, 1.0, "bf16")
    n = ref.logprob_entropy(d["h"], d["W"], d["targets"], None, 1.0, "bf16")
    for k in ("logp", "ent", "lse", "ez"):
        np.testing.assert_allclose(c[k], n[k], rtol=1e-12, atol=1e-11)


def test_c_and_numpy_agree_packed_fp16():
    w = workloads.WORKLOADS[2].scaled(T=3000, H=64, V=1000)
    d = workloads.make(w)
    rows = d["row_idx"].numpy()
    assert 0 < rows.shape[0] < 3000
    c = coracle.logprob_entropy(d["h"], d["W"], d["targets"], rows, 1.0, "fp16")
    n = ref.logprob_entropy(d["h"], d["W"], d["targets"], rows, 1.0, "fp16")
    for k in ("logp", "ent"):
        np.testing.assert_allclose(c[k], n[k], rtol=1e-12, atol=1e-11)


def test_c_and_numpy_agree_kl():
    w = workloads.WORKLOADS[3].scaled(T=40, H=64, V=900)
    d = workloads.make(w)
    a = coracle.kl(d["h_s"], d["W_s"], d["h_t"], d["W_t"], None, "bf16")
    b = ref.kl(d["h_s"], d["W_s"], d["h_t"], d["W_t"], None, "bf16")
    np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-13)


# --------------------------------------------------------------------------
# K targets per row

def test_k_targets_reduce_to_single_targets():
    d = _random_case(16, T=20, V=700)
    rng = np.random.default_rng(16)
    tk = rng.integers(0, 700, size=(20, 5))
    rows = np.array([3, 19, 0, 7, 7])
    o = coracle.logprob_k(d["h"], d["W"], tk, rows, 0.7, "bf16")
    assert o["rc"] == 0
    for k in range(5):
        single = coracle.logprob_entropy(d["h"], d["W"], tk[:, k], rows, 0.7, "bf16")
        np.testing.assert_array_equal(o["logp"][:, k], single["logp"])
        np.testing.assert_array_equal(o["ent"], single["ent"])


def test_k_targets_over_the_whole_vocabulary_sum_to_one():
    """With every token as a candidate, exp(logp) is the softmax: it sums to 1."""
    d = _random_case(17, T=6, H=16, V=300)
    tk = np.tile(np.arange(300), (6, 1))
    o = coracle.logprob_k(d["h"], d["W"], tk, None, 0.9, "bf16")
    np.testing.assert_allclose(np.exp(o["logp"]).sum(axis=1), 1.0, atol=1e-12)
    # the entropy is the entropy of that distribution
    p = np.exp(o["logp"])
    np.testing.assert_allclose(-(p * o["logp"]).sum(axis=1), o["ent"], atol=1e-11)


def test_k_targets_bad_candidate_is_nan():
    d = _random_case(18, T=4, V=100)
    tk = np.array([[1, 2], [3, 100], [5, -1], [7, 8]])
    o = coracle.logprob_k(d["h"], d["W"], tk, None, 1.0, "bf16")
    assert o["rc"] == -1
    assert np.isnan(o["logp"][1, 1]) and np.isnan(o["logp"][2, 1])
    assert np.isfinite(o["logp"][[0, 3]]).all() and np.isfinite(o["logp"][[1, 2], 0]).all()


# --------------------------------------------------------------------------
# sampling support (the per-row vocabulary mask of calculate_log_probs_and_entropy)

def _support_case(seed, T=10, H=16, V=150, j=1, force=True, dtype="bf16"):
    d = _random_case(seed, T=T, H=H, V=V, dtype=dtype)
    tg = d["targets"].numpy()
    sup = workloads.support_words(T, V, j, seed, targets=tg if force else None)
    return d, tg, sup


def test_support_of_every_token_is_the_unrestricted_result():
    d, tg, sup = _support_case(40, j=0)
    rows = np.array([9, 0, 4, 4])
    for f, g in ((coracle.logprob_entropy_support, coracle.logprob_entropy),
                 (lambda *a: ref.logprob_entropy(*a[:4], a[5], a[6], support=a[4]),
                  ref.logprob_entropy)):
        a = f(d["h"], d["W"], tg, rows, sup, 0.8, "bf16")
        b = g(d["h"], d["W"], tg, rows, 0.8, "bf16")
        for k in ("logp", "ent", "lse", "ez"):
            np.testing.assert_allclose(a[k], b[k], rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("j", [1, 3])
def test_support_is_the_problem_on_the_kept_vocabulary(j):
    """Restricting to S is the unrestricted problem on the vocabulary rows W[S]
    with the target renumbered: row by row, with the plain oracle."""
    d, tg, sup = _support_case(41 + j, j=j)
    Wd = ref.decode(d["W"], "bf16")
    keep = ref.support_bits(sup, np.arange(10), 150)
    got = coracle.logprob_entropy_support(d["h"], d["W"], tg, None, sup, 0.7, "bf16")
    assert got["rc"] == 0
    for r in range(10):
        S = np.nonzero(keep[r])[0]
        t_new = np.full(10, 0)
        t_new[r] = int(np.searchsorted(S, tg[r]))
        assert S[t_new[r]] == tg[r]
        sub = coracle.logprob_entropy(ref.decode(d["h"], "bf16"), Wd[S], t_new, [r], 0.7, "f64")
        for k in ("logp", "ent", "lse", "ez"):
            assert got[k][r] == pytest.approx(sub[k][0], rel=1e-13, abs=1e-13), (r, k)


def _dec_forward_support(h, W, tg, rows, keep, tau):
    getcontext().prec = 50
    out = []
    for r in rows:
        S = [v for v in range(W.shape[0]) if keep[r, v]]
        z = {v: sum(Decimal(float(h[r, k])) * Decimal(float(W[v, k])) for k in range(h.shape[1]))
             / Decimal(repr(tau)) for v in S}
        lse = sum((x.exp() for x in z.values()), Decimal(0)).ln()
        ez = sum(((x - lse).exp() * x for x in z.values()), Decimal(0))
        out.append((float(z[tg[r]] - lse), float(lse - ez), float(lse), float(ez)))
    return np.array(out)


@pytest.mark.parametrize("tau", [0.7, 1.3])
def test_support_brute_force(tau):
    d, tg, sup = _support_case(44, T=6, H=11, V=45, j=1)
    rows = np.array([5, 2, 0, 2])
    keep = ref.support_bits(sup, np.arange(6), 45)
    want = _dec_forward_support(ref.decode(d["h"], "bf16"), ref.decode(d["W"], "bf16"), tg, rows,
                                keep, tau)
    c = coracle.logprob_entropy_support(d["h"], d["W"], tg, rows, sup, tau, "bf16")
    n = ref.logprob_entropy(d["h"], d["W"], tg, rows, tau, "bf16", support=sup)
    for o in (c, n):
        got = np.stack([o["logp"], o["ent"], o["lse"], o["ez"]], axis=1)
        np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)


def test_support_singleton_and_pair_closed_forms():
    rng = np.random.default_rng(45)
    T, H, V = 4, 6, 70
    h, W = rng.standard_normal((T, H)), rng.standard_normal((V, H))
    tg = np.array([3, 40, 69, 0])
    other = np.array([64, 41, 1, 33])
    sup = np.zeros((T, 3), dtype=np.uint32)
    for r in range(T):
        sup[r, tg[r] // 32] |= np.uint32(1 << (tg[r] % 32))
    one = coracle.logprob_entropy_support(h, W, tg, None, sup.view(np.int32), 0.9, "f64")
    assert np.all(one["logp"] == 0.0) and np.all(one["ent"] == 0.0)
    for r in range(T):
        sup[r, other[r] // 32] |= np.uint32(1 << (other[r] % 32))
    two = coracle.logprob_entropy_support(h, W, tg, None, sup.view(np.int32), 0.9, "f64")
    for r in range(T):
        dz = (h[r] @ W[other[r]] - h[r] @ W[tg[r]]) / 0.9
        q = 1 / (1 + math.exp(dz))                  # probability of the target
        assert two["logp"][r] == pytest.approx(math.log(q), abs=1e-14)
        assert two["ent"][r] == pytest.approx(-q * math.log(q) - (1 - q) * math.log(1 - q),
                                              abs=1e-14)


def test_support_target_off_support_and_empty_support():
    d, tg, sup = _support_case(46, T=5, V=100, j=2)
    words = sup.view(np.uint32).copy()
    words[1, tg[1] // 32] &= ~np.uint32(1 << (tg[1] % 32))     # target of row 1 off
    words[3, :] = 0                                             # row 3: empty support
    s = words.view(np.int32)
    c = coracle.logprob_entropy_support(d["h"], d["W"], tg, None, s, 1.0, "bf16")
    n = ref.logprob_entropy(d["h"], d["W"], tg, None, 1.0, "bf16", support=s)
    assert c["rc"] == -1
    for o in (c, n):
        assert o["logp"][1] == -np.inf and np.isfinite(o["ent"][1])
        assert np.isnan(o["logp"][3]) and np.isnan(o["ent"][3])
        assert np.isfinite(o["logp"][[0, 2, 4]]).all()
    np.testing.assert_allclose(c["ent"][[0, 1, 2, 4]], n["ent"][[0, 1, 2, 4]], rtol=1e-12)


def _loss_support(h, W, tg, rows, sup, tau, g1, g2):
    o = coracle.logprob_entropy_support(h, W, tg, rows, sup, tau, "f64")
    return float(np.sum(g1 * o["logp"] + g2 * o["ent"]))


@pytest.mark.parametrize("tau", [0.7, 1.0])
def test_support_backward_matches_finite_differences(tau):
    rng = np.random.default_rng(47)
    T, H, V = 5, 4, 40
    h = rng.standard_normal((T, H))
    W = rng.standard_normal((V, H)) * 0.7
    tg = rng.integers(0, V, size=T)
    sup = workloads.support_words(T, V, 1, 47, targets=tg)
    rows = np.array([4, 0, 2])
    g1, g2 = rng.standard_normal(3), rng.standard_normal(3)
    dh_rows, dW = coracle.backward_support(h, W, tg, rows, sup, tau, g1, g2, "f64")
    dh = coracle.scatter_rows(dh_rows, rows, T)
    eps = 1e-6
    num_h = np.zeros_like(h)
    for r in range(T):
        for k in range(H):
            hp, hm = h.copy(), h.copy()
            hp[r, k] += eps
            hm[r, k] -= eps
            num_h[r, k] = (_loss_support(hp, W, tg, rows, sup, tau, g1, g2)
                           - _loss_support(hm, W, tg, rows, sup, tau, g1, g2)) / (2 * eps)
    num_W = np.zeros_like(W)
    for v in range(V):
        for k in range(H):
            Wp, Wm = W.copy(), W.copy()
            Wp[v, k] += eps
            Wm[v, k] -= eps
            num_W[v, k] = (_loss_support(h, Wp, tg, rows, sup, tau, g1, g2)
                           - _loss_support(h, Wm, tg, rows, sup, tau, g1, g2)) / (2 * eps)
    assert np.linalg.norm(dh - num_h) <= 1e-6 * np.linalg.norm(num_h)
    assert np.linalg.norm(dW - num_W) <= 1e-6 * np.linalg.norm(num_W)
    # vocabulary rows outside every scored row's support get no gradient
    keep = ref.support_bits(sup, rows, V).any(axis=0)
    assert np.all(dW[~keep] == 0.0) and (~keep).any()
    rdh, rdW = ref.backward(h, W, tg, rows, tau, g1, g2, "f64", support=sup)
    np.testing.assert_allclose(rdh, dh_rows, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(rdW, dW, rtol=1e-10, atol=1e-12)


def test_support_backward_columns_sum_to_zero():
    """On the support, sum_v G_rv = 0 still holds (targets inside it), so the
    column sums of dW vanish."""
    d, tg, sup = _support_case(48, T=12, H=20, V=300, j=2)
    rows = np.arange(12)
    rng = np.random.default_rng(48)
    _, dW = coracle.backward_support(d["h"], d["W"], tg, rows, sup, 0.7, rng.standard_normal(12),
                                     rng.standard_normal(12), "bf16")
    scale = np.abs(dW).sum(axis=0)
    assert np.all(np.abs(dW.sum(axis=0)) <= 1e-12 * scale + 1e-15)


def test_support_c_and_numpy_agree_config0():
    d = workloads.make(0)
    tg = d["targets"].numpy()
    sup = workloads.support_words(256, 8192, 2, 0, targets=tg, ld=260)
    rows = workloads.sample_rows(256, 40, seed=3)
    c = coracle.logprob_entropy_support(d["h"], d["W"], tg, rows, sup, 1.0, "bf16")
    n = ref.logprob_entropy(d["h"], d["W"], tg, rows, 1.0, "bf16", support=sup)
    for k in ("logp", "ent", "lse", "ez"):
        np.testing.assert_allclose(c[k], n[k], rtol=1e-10, atol=1e-12)
    g1 = np.linspace(-1, 1, 40)
    g2 = np.linspace(1, -0.5, 40)
    vs = np.array([0, 5, 8191, int(tg[rows[0]])])
    cdh, cdW = coracle.backward_support(d["h"], d["W"], tg, rows[:6], sup, 1.0, g1[:6], g2[:6],
                                        "bf16", vsel=vs)
    ndh, ndW = ref.backward(d["h"], d["W"], tg, rows[:6], 1.0, g1[:6], g2[:6], "bf16",
                            vsel=vs, support=sup)
    np.testing.assert_allclose(cdh, ndh, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(cdW, ndW, rtol=1e-9, atol=1e-12)


# --------------------------------------------------------------------------
# MXFP4 teacher head (OCP Microscaling FP4: E2M1 elements, E8M0 block scales)

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_mxfp4_decoding_is_the_e2m1_table_times_the_block_scale():
    V, H = 3, 64
    packed = np.zeros((1, 256, 32), np.uint8)
    scales = np.zeros((1, 256, 2), np.uint8)
    codes = np.arange(64) % 16                      # every nibble, twice per row
    for v in range(V):
        packed[0, v] = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
        scales[0, v] = (127 + v - 1, 127 + 3 * v)    # 2^(v-1) and 2^(3v)
    for deq in (coracle.mxfp4_dequantize(packed, scales, V),
                ref.mxfp4_dequantize(packed, scales, V)):
        for v in range(V):
            for k in range(64):
                c = codes[k]
                want = (-1.0 if c & 8 else 1.0) * E2M1[c & 7] * 2.0 ** (
                    (v - 1) if k < 32 else 3 * v)
                assert deq[v, k] == want, (v, k)


def test_mxfp4_grid_values_round_trip_exactly():
    """A block of grid values whose largest magnitude is 4 or 6 (times 2^e)
    gets scale code e + 127 and is stored exactly."""
    rng = np.random.default_rng(70)
    V, H = 40, 128
    mags = np.array(E2M1)
    e = rng.integers(-20, 10, size=(V, H // 32))
    top = rng.choice([4.0, 6.0], size=(V, H // 32))
    x = rng.choice(mags, size=(V, H // 32, 32)) * rng.choice([-1.0, 1.0], size=(V, H // 32, 32))
    x[:, :, 0] = top
    W = (x * np.ldexp(1.0, e)[:, :, None]).reshape(V, H)
    for q in (coracle.mxfp4_quantize(W, "f64"), ref.mxfp4_quantize(W, "f64")):
        assert np.array_equal(q[1][:, :V, :].transpose(1, 0, 2).reshape(V, -1), e + 127)
        assert np.array_equal(coracle.mxfp4_dequantize(*q, V), W)


def test_mxfp4_rounding_is_nearest_with_ties_to_even_and_saturation():
    rng = np.random.default_rng(71)
    V, H = 64, 256
    W = rng.standard_normal((V, H)) * np.exp(rng.uniform(-3, 3, size=(V, 1)))
    W[0, :32] = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 5.5, 7.0] + [0.0] * 22 + [7.9])
    W[1, :32] = 0.0
    packed, scales = coracle.mxfp4_quantize(W, "f64")
    deq = coracle.mxfp4_dequantize(packed, scales, V)
    code = scales[:, :V, :].transpose(1, 0, 2).reshape(V, H // 32).astype(np.int64)
    # the block scale: 2^(floor(log2 max|x|) - 2)
    amax = np.abs(W.reshape(V, H // 32, 32)).max(axis=2)
    want_code = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1))) - 2 + 127, 0)
    assert np.array_equal(code, want_code)
    unit = np.repeat(np.ldexp(1.0, code - 127), 32, axis=1)
    a = np.abs(W) / unit
    grid = np.array(E2M1)
    for v in range(V):
        for k in range(H):
            got = abs(deq[v, k]) / unit[v, k]
            d = np.abs(grid - min(a[v, k], 6.0))
            best = d.min()
            ties = np.nonzero(d == best)[0]
            want = grid[ties[0]] if len(ties) == 1 else grid[[t for t in ties if t % 2 == 0][0]]
            assert got == want, (v, k, a[v, k], got)
            if got != 0:
                assert np.sign(deq[v, k]) == np.sign(W[v, k])
    # the printed tie cases, in units of the block scale (max 7.9 -> scale 1)
    assert code[0, 0] == 127
    assert deq[0, :9].tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0]
    assert np.all(deq[1, :32] == 0.0) and code[1, 0] == 0


def test_mxfp4_c_and_numpy_quantisers_agree():
    w = workloads.WORKLOADS[3].scaled(T=4, H=256, V=700, seed=72)
    d = workloads.make(w)
    for m in (d["W_t"], d["W_s"]):
        pc, sc = coracle.mxfp4_quantize(m, "bf16")
        pn, sn = ref.mxfp4_quantize(m, "bf16")
        assert np.array_equal(pc, pn) and np.array_equal(sc, sn)
        assert np.all(pc[:, 700:, :] == 0) and np.all(sc[:, 700:, :] == 0)   # padding rows


def test_kl_with_mxfp4_teacher_is_kl_on_the_decoded_weights():
    w = workloads.WORKLOADS[3].scaled(T=10, H=128, V=400, seed=73)
    d = workloads.make(w)
    packed, scales = coracle.mxfp4_quantize(d["W_t"], "bf16")
    Wt = coracle.mxfp4_dequantize(packed, scales, 400)
    rows = np.array([9, 0, 4])
    got = coracle.kl_mxfp4(d["h_s"], d["W_s"], d["h_t"], packed, scales, rows, "bf16")
    dec = [ref.decode(d[k], "bf16") for k in ("h_s", "W_s", "h_t")]
    want = coracle.kl(dec[0], dec[1], dec[2], Wt, rows, "f64")
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(ref.kl_mxfp4(d["h_s"], d["W_s"], d["h_t"], packed, scales, rows,
                                            "bf16"), want, rtol=1e-10, atol=1e-13)
    # the teacher's quantisation moves the KL, but not by much at these sizes
    plain = coracle.kl(d["h_s"], d["W_s"], d["h_t"], d["W_t"], rows, "bf16")
    assert np.all(np.abs(got - plain) < 0.1 * plain)


# --------------------------------------------------------------------------
# MXFP8 teacher rows (OCP Microscaling FP8: E4M3 elements, E8M0 block scales),
# the hidden-state side of the block-scaled teacher path

def test_e4m3_decoding_every_code():
    """Both oracle decoders give the E4M3 value of every code: 1 sign, 4
    exponent bits (bias 7), 3 mantissa bits, subnormals below exponent field
    1, NaN at 0x7F / 0xFF, 448 the largest finite value.  Checked against the
    format's definition written out here and against torch.float8_e4m3fn."""
    want = []
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            want.append(float("nan"))
            continue
        v = (1 + m / 8) * 2.0 ** (e - 7) if e else (m / 8) * 2.0 ** -6
        want.append(-v if s else v)
    want = np.array(want)
    lib_vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(want)
    for got in (np.array([coracle.e4m3_value(c) for c in range(256)]), ref.e4m3_values(), lib_vals):
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan], want[~nan])
    assert want[0x38] == 1.0 and want[0x7E] == 448.0 and want[0x01] == 2.0 ** -9
    assert want[0x08] == 2.0 ** -6 and want[0xB8] == -1.0 and want[0x77] == 240.0


def test_mxfp8_scale_is_the_block_maximum_exponent_minus_8():
    rng = np.random.default_rng(80)
    R, H = 32, 256
    X = rng.standard_normal((R, H)) * np.exp(rng.uniform(-20, 20, size=(R, 1)))
    X[3, 32:64] = 0.0
    for codes, scales in (coracle.mxfp8_quantize(X, "f64"), ref.mxfp8_quantize(X, "f64")):
        amax = np.abs(X.reshape(R, H // 32, 32)).max(axis=2)
        want = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1))) - 8 + 127, 0)
        assert np.array_equal(scales.astype(np.int64), want)
        assert scales[3, 1] == 0 and np.all(codes[3, 32:64] == 0)


def test_mxfp8_rounding_matches_torch_e4m3_below_saturation():
    """Inside the block's scale unit the element is the E4M3 value nearest to
    x / 2^(scale - 127), ties to even; torch's float8_e4m3fn conversion, an
    independent round-to-nearest-even, agrees wherever it does not overflow
    (x / unit <= 464).  Above that the oracle saturates at 448."""
    rng = np.random.default_rng(81)
    R, H = 64, 256
    X = rng.standard_normal((R, H))
    # exact midpoints between neighbouring codes, in units of the scale
    vals = ref.e4m3_values()[:0x7F]
    mids = (vals[:-1] + vals[1:]) / 2
    X[0, :32] = 0.0
    X[0, 0] = 448.0                                 # scale 2^0
    X[0, 1:32] = mids[rng.choice(len(mids), 31)]
    X[1, :32] = [500.0] + [470.0, 464.0, 463.0, 449.0] + [1.0] * 27   # scale 2^0, saturation
    codes, scales = coracle.mxfp8_quantize(X, "f64")
    deq = coracle.mxfp8_dequantize(codes, scales)
    unit = np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=1)
    a = X / unit
    ok = np.abs(a) <= 464.0
    lib = torch.from_numpy(a[ok]).float().to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(deq[ok] / unit[ok], lib)
    assert deq[1, :5].tolist() == [448.0, 448.0, 448.0, 448.0, 448.0]
    assert np.array_equal(codes, ref.mxfp8_quantize(X, "f64")[0])


def test_mxfp8_grid_values_round_trip_exactly():
    """A block of E4M3 values whose largest is 448 (times 2^k) gets scale
    code k + 127 and is stored exactly."""
    rng = np.random.default_rng(82)
    R, H = 24, 128
    vals = ref.e4m3_values()[:0x7F]
    k = rng.integers(-60, 40, size=(R, H // 32))
    x = rng.choice(vals, size=(R, H // 32, 32)) * rng.choice([-1.0, 1.0], size=(R, H // 32, 32))
    x[:, :, 0] = 448.0
    X = (x * np.ldexp(1.0, k)[:, :, None]).reshape(R, H)
    for codes, scales in (coracle.mxfp8_quantize(X, "f64"), ref.mxfp8_quantize(X, "f64")):
        assert np.array_equal(scales.astype(np.int64), k + 127)
        assert np.array_equal(coracle.mxfp8_dequantize(codes, scales), X)


def test_mxfp8_c_and_numpy_quantisers_agree():
    w = workloads.WORKLOADS[3].scaled(T=200, H=256, V=64, seed=83)
    d = workloads.make(w)
    for m in (d["h_t"], d["h_s"]):
        cc, sc = coracle.mxfp8_quantize(m, "bf16")
        cn, sn = ref.mxfp8_quantize(m, "bf16")
        assert np.array_equal(cc, cn) and np.array_equal(sc, sn)
    # signs, zeros (stored as +0) and values far below the block maximum
    x = np.array([[-0.0, 0.0, -1e-30, 1e-30, 3.0, -3.0, 2.0 ** -140, -7.5] * 4])
    cc, sc = coracle.mxfp8_quantize(x, "f64")
    assert np.array_equal(cc, ref.mxfp8_quantize(x, "f64")[0])
    assert cc[0, 0] == 0 and cc[0, 2] == 0 and cc[0, 6] == 0


def test_kl_block_scaled_teacher_on_the_grid_is_the_mxfp4_kl():
    """Teacher rows already on the MXFP8 grid are not changed by the
    quantisation, so the block-scaled KL equals the MXFP4-teacher KL on the
    same (decoded) inputs; with the student equal to the teacher it is 0."""
    w = workloads.WORKLOADS[3].scaled(T=12, H=128, V=300, seed=84)
    d = workloads.make(w)
    ht = coracle.mxfp8_dequantize(*coracle.mxfp8_quantize(d["h_t"], "bf16"))
    ht_bits = _bits(ht, "bf16").reshape(ht.shape)                 # exact in bf16
    assert np.array_equal(ref.decode(ht_bits, "bf16"), ht)
    packed, scales = coracle.mxfp4_quantize(d["W_t"], "bf16")
    rows = np.array([11, 0, 5, 5])
    hs = _bits(ref.decode(d["h_s"], "bf16"), "bf16").reshape(ht.shape)
    got = coracle.kl_mx(hs, d["W_s"], ht_bits, packed, scales, rows, "bf16")
    want = coracle.kl_mxfp4(hs, d["W_s"], ht_bits, packed, scales, rows, "bf16")
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(ref.kl_mx(hs, d["W_s"], ht_bits, packed, scales, rows, "bf16"),
                               want, rtol=1e-10, atol=1e-13)
    # student = teacher: h_s on the MXFP8 grid, W_s the decoded MXFP4 head
    Wt = coracle.mxfp4_dequantize(packed, scales, 300)
    Ws_bits = _bits(Wt, "bf16").reshape(Wt.shape)
    same = coracle.kl_mx(ht_bits, Ws_bits, ht_bits, packed, scales, rows, "bf16")
    assert np.all(np.abs(same) <= 1e-13)


def test_kl_block_scaled_teacher_c_and_numpy_agree():
    w = workloads.WORKLOADS[3].scaled(T=20, H=256, V=500, seed=85)
    d = workloads.make(w)
    packed, scales = coracle.mxfp4_quantize(d["W_t"], "bf16")
    rows = np.array([19, 3, 7, 0])
    got = coracle.kl_mx(d["h_s"], d["W_s"], d["h_t"], packed, scales, rows, "bf16")
    np.testing.assert_allclose(ref.kl_mx(d["h_s"], d["W_s"], d["h_t"], packed, scales, rows,
                                         "bf16"), got, rtol=1e-10, atol=1e-13)
    assert np.all(got >= 0)
    # the teacher rows' quantisation moves the KL, but not by much
    base = coracle.kl_mxfp4(d["h_s"], d["W_s"], d["h_t"], packed, scales, rows, "bf16")
    assert np.all(np.abs(got - base) < 0.2 * base)


# --------------------------------------------------------------------------
# Log-prob and entropy on the block-scaled path (an inference-only forward,
# e.g. the reference model's log-probs): MXFP8 rows x MXFP4 head

def test_logprob_entropy_block_scaled_is_the_plain_forward_on_the_decoded_operands():
    """Rows on the MXFP8 grid are left alone by the quantisation and the head
    is its decoded MXFP4 values, so the block-scaled forward equals the plain
    forward on those values; rows off the grid score as their MXFP8 values."""
    w = workloads.WORKLOADS[1].scaled(T=14, H=128, V=300, seed=86)
    d = workloads.make(w)
    packed, scales = coracle.mxfp4_quantize(d["W"], "bf16")
    Wd = coracle.mxfp4_dequantize(packed, scales, 300)
    Wd_bits = _bits(Wd, "bf16").reshape(Wd.shape)                  # exact in bf16
    assert np.array_equal(ref.decode(Wd_bits, "bf16"), Wd)
    hq = coracle.mxfp8_dequantize(*coracle.mxfp8_quantize(d["h"], "bf16"))
    hq_bits = _bits(hq, "bf16").reshape(hq.shape)
    assert np.array_equal(ref.decode(hq_bits, "bf16"), hq)
    rows = np.array([13, 0, 6, 6, 2])
    tg = d["targets"]
    for h in (hq_bits, d["h"]):   # on the grid, then the raw rows
        got = coracle.logprob_entropy_mx(h, packed, scales, 300, tg, rows, 0.7, "bf16")
        want = coracle.logprob_entropy(hq_bits, Wd_bits, tg, rows, 0.7, "bf16")
        for k in ("logp", "ent", "lse", "ez"):
            np.testing.assert_allclose(got[k], want[k], rtol=1e-13, atol=1e-13)
        assert got["rc"] == 0
    # the quantisation moves the scores, but not by much at these sizes
    plain = coracle.logprob_entropy(d["h"], d["W"], tg, rows, 0.7, "bf16")
    assert np.all(np.abs(got["ent"] - plain["ent"]) < 0.05 * plain["ent"])


def test_logprob_entropy_block_scaled_closed_forms_and_bounds():
    """A zero head gives logp = -ln V and entropy = ln V; every row keeps
    logp <= 0 and 0 <= entropy <= ln V; a bad row index gives NaN."""
    w = workloads.WORKLOADS[1].scaled(T=9, H=64, V=257, seed=87)
    d = workloads.make(w)
    zero = np.zeros((257, 64))
    packed, scales = coracle.mxfp4_quantize(zero, "f64")
    assert not packed.any() and not scales.any()
    out = coracle.logprob_entropy_mx(d["h"], packed, scales, 257, d["targets"], None, 1.3, "bf16")
    np.testing.assert_allclose(out["logp"], -LN(257), rtol=0, atol=1e-12)
    np.testing.assert_allclose(out["ent"], LN(257), rtol=0, atol=1e-12)
    packed, scales = coracle.mxfp4_quantize(d["W"], "bf16")
    rows = np.array([8, -1, 3, 9])
    out = coracle.logprob_entropy_mx(d["h"], packed, scales, 257, d["targets"], rows, 0.7, "bf16")
    assert out["rc"] == -1
    ok = np.array([True, False, True, False])
    assert np.all(np.isnan(out["logp"][~ok])) and np.all(np.isnan(out["ent"][~ok]))
    assert np.all(out["logp"][ok] <= 0)
    assert np.all((out["ent"][ok] >= 0) & (out["ent"][ok] <= LN(257)))


def test_logprob_entropy_block_scaled_c_and_numpy_agree():
    w = workloads.WORKLOADS[1].scaled(T=40, H=256, V=700, seed=88)
    d = workloads.make(w)
    packed, scales = coracle.mxfp4_quantize(d["W"], "bf16")
    rows = np.array([39, 3, 7, 0, 3, 22])
    got = coracle.logprob_entropy_mx(d["h"], packed, scales, 700, d["targets"], rows, 0.7, "bf16")
    want = ref.logprob_entropy_mx(d["h"], packed, scales, 700, d["targets"], rows, 0.7, "bf16")
    for k in ("logp", "ent", "lse", "ez"):
        np.testing.assert_allclose(got[k], want[k], rtol=1e-10, atol=1e-11)
    got16 = coracle.logprob_entropy_mx(_bits(ref.decode(d["h"], "bf16"), "fp16").reshape(40, 256),
                                       packed, scales, 700, d["targets"], rows, 1.0, "fp16")
    want16 = ref.logprob_entropy_mx(_bits(ref.decode(d["h"], "bf16"), "fp16").reshape(40, 256),
                                    packed, scales, 700, d["targets"], rows, 1.0, "fp16")
    np.testing.assert_allclose(got16["logp"], want16["logp"], rtol=1e-10, atol=1e-11)
