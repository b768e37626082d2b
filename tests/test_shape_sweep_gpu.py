"""Seeded sweep of random shapes through the forward, the KL and the
backward, each compared with the float64 oracle.

The fixed-shape parity tests pick their ragged cases by hand.  This sweep
draws 48 more from one seeded generator: rows T in [1, 700], hidden size H a
multiple of 8 in [8, 1024], vocabulary V from 1 to 40,000 (log-uniform),
bf16 or fp16, a temperature in [0.3, 3], and either all rows or a random
row selection (unsorted, with repeats).  So tails of every kind fall at
random places: a part of a 128-row tile, of a 64-wide K block, of a
32-column chunk and of a 512-column vocabulary tile, and the few-rows path
(n <= 128) against the pair path.  Each case is small enough for the C
oracle to finish in about a second.  The same cases also run the K-target
forward, the forward and backward under a sampling support, the KL with an
MXFP4 teacher head, decoded and on the block-scaled tensor cores, and the
forward on the block-scaled tensor cores.

Tolerances are those of the fixed-shape tests: |d logp|, |d ent|, |d KL|
<= 1e-3 absolute; gradients within 1e-2 relative (Frobenius, and every
element within 1e-2 of the largest).
"""
import numpy as np
import pytest
import torch

import entropy_tcgen05_vocab_gb300 as flp
import workloads
from oracle import coracle

pytestmark = pytest.mark.gpu
TOL = 1e-3
RTOL = 1e-2
N_CASES = 48
MAX_WORK = 6e8   # n * V * H per case, so the oracle stays near a second


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    flp.build()
    flp.lib()


def _draw(case):
    """Shape, dtype, temperature and row selection of sweep case ``case``."""
    r = np.random.Generator(np.random.PCG64([2026, case]))
    while True:
        T = int(r.integers(1, 701))
        H = 8 * int(r.integers(1, 129))
        V = int(np.exp(r.uniform(0.0, np.log(40000.0)))) + 1
        if T * V * H <= MAX_WORK:
            break
    dtype = "bf16" if r.random() < 0.6 else "fp16"
    tau = float(np.round(r.uniform(0.3, 3.0), 3))
    if r.random() < 0.4:
        rows = None
    else:
        n = int(r.integers(1, 2 * T + 1))
        rows = r.integers(0, T, size=n).astype(np.int64)
    return T, H, V, dtype, tau, rows, int(r.integers(0, 2**31))


def _scaled(kind, T, H, V, dtype, tau, seed):
    base = {"fwd": 0, "kl": 3, "bwd": 4}[kind]
    w = workloads.WORKLOADS[base].scaled(T=T, H=H, V=V, dtype=dtype, tau=tau, seed=seed,
                                         w_std=0.06, rows="all", targets="uniform")
    return workloads.make(w, device="cuda")


def _abs(got, want, what):
    g = got.detach().cpu().double().numpy()
    assert np.all(np.isfinite(g)), what + ": non-finite output"
    err = np.abs(g - want)
    assert err.max() <= TOL, "%s: max |diff| %.3e at %d" % (what, err.max(), int(err.argmax()))


def _rel(got, want, what):
    g = got.detach().cpu().double().numpy()
    assert np.all(np.isfinite(g)), what + ": non-finite"
    fro = np.linalg.norm(g - want) / max(np.linalg.norm(want), 1e-30)
    ele = np.abs(g - want).max() / max(np.abs(want).max(), 1e-30)
    assert fro <= RTOL and ele <= RTOL, "%s: rel Frobenius %.2e, rel max %.2e" % (what, fro, ele)


def _rel_or_zero(got, want, what):
    if np.abs(want).max() < 1e-6:   # e.g. a one-token vocabulary: every gradient is zero
        g = got.detach().cpu().double().numpy()
        assert np.all(np.isfinite(g)) and np.abs(g).max() <= 1e-5, what + ": expected zeros"
        return
    _rel(got, want, what)


CASES = [_draw(c) for c in range(N_CASES)]


def _id(c):
    T, H, V, dtype, tau, rows, _ = c
    return "T%d-H%d-V%d-%s-tau%g-%s" % (T, H, V, dtype, tau,
                                        "all" if rows is None else "n%d" % len(rows))


@pytest.mark.parametrize("case", CASES, ids=[_id(c) for c in CASES])
def test_forward_sweep(case):
    T, H, V, dtype, tau, rows, seed = case
    d = _scaled("fwd", T, H, V, dtype, tau, seed)
    ri = None if rows is None else torch.from_numpy(rows).cuda()
    logp, ent, lse, ez = flp.logprob_entropy(d["h"], d["W"], d["targets"], ri, tau,
                                             return_stats=True)
    torch.cuda.synchronize()
    o = coracle.logprob_entropy(d["h"].cpu(), d["W"].cpu(), d["targets"].cpu().numpy(), rows,
                                tau, dtype)
    _abs(logp, o["logp"], "logp")
    _abs(ent, o["ent"], "ent")
    _abs(lse, o["lse"], "lse")


@pytest.mark.parametrize("case", CASES[::2], ids=[_id(c) for c in CASES[::2]])
def test_kl_sweep(case):
    T, H, V, dtype, _, rows, seed = case
    d = _scaled("kl", T, H, V, dtype, 1.0, seed)
    ri = None if rows is None else torch.from_numpy(rows).cuda()
    kl = flp.kl_divergence(d["h_s"], d["W_s"], d["h_t"], d["W_t"], ri)
    torch.cuda.synchronize()
    want = coracle.kl(d["h_s"].cpu(), d["W_s"].cpu(), d["h_t"].cpu(), d["W_t"].cpu(), rows, dtype)
    _abs(kl, want, "kl")


@pytest.mark.parametrize("case", CASES[1::2], ids=[_id(c) for c in CASES[1::2]])
def test_backward_sweep(case):
    T, H, V, dtype, tau, rows, seed = case
    d = _scaled("bwd", T, H, V, dtype, tau, seed)
    n = T if rows is None else len(rows)
    g = np.random.Generator(np.random.PCG64([seed, 7]))
    g1 = torch.from_numpy(g.standard_normal(n, dtype=np.float32)).cuda()
    g2 = torch.from_numpy(g.standard_normal(n, dtype=np.float32)).cuda()
    ri = None if rows is None else torch.from_numpy(rows).cuda()
    dh, dW = flp.backward(d["h"], d["W"], d["targets"], ri, tau, g1, g2)
    torch.cuda.synchronize()
    dh_rows, ref_dW = coracle.backward(d["h"].cpu(), d["W"].cpu(), d["targets"].cpu().numpy(),
                                       rows, tau, g1.cpu().numpy(), g2.cpu().numpy(), dtype)
    ref_dh = coracle.scatter_rows(dh_rows, np.arange(T) if rows is None else rows, T)
    _rel_or_zero(dh, ref_dh, "dh")
    _rel_or_zero(dW, ref_dW, "dW")


def _extra(case, k):
    """A second seeded draw per case for the widened calls (K, support density)."""
    return np.random.Generator(np.random.PCG64([2027, case[-1] % (2**31), k]))


@pytest.mark.parametrize("case", CASES[::3], ids=[_id(c) for c in CASES[::3]])
def test_k_targets_sweep(case):
    T, H, V, dtype, tau, rows, seed = case
    d = _scaled("fwd", T, H, V, dtype, tau, seed)
    r = _extra(case, 1)
    K = int(r.integers(1, 9))
    tk = torch.from_numpy(r.integers(0, V, size=(T, K)).astype(np.int64))
    ri = None if rows is None else torch.from_numpy(rows).cuda()
    logp, ent = flp.logprob_entropy_k(d["h"], d["W"], tk.cuda(), ri, tau)
    torch.cuda.synchronize()
    o = coracle.logprob_k(d["h"].cpu(), d["W"].cpu(), tk.numpy(), rows, tau, dtype)
    _abs(logp, o["logp"], "logp[K=%d]" % K)
    _abs(ent, o["ent"], "ent")


@pytest.mark.parametrize("case", CASES[1::3], ids=[_id(c) for c in CASES[1::3]])
def test_support_forward_sweep(case):
    T, H, V, dtype, tau, rows, seed = case
    d = _scaled("fwd", T, H, V, dtype, tau, seed)
    j = int(_extra(case, 2).integers(0, 4))
    sup = workloads.support_words(T, V, j, seed % (2**31), targets=d["targets"].cpu().numpy())
    ri = None if rows is None else torch.from_numpy(rows).cuda()
    logp, ent = flp.logprob_entropy(d["h"], d["W"], d["targets"], ri, tau,
                                    support=torch.from_numpy(sup).cuda())
    torch.cuda.synchronize()
    o = coracle.logprob_entropy_support(d["h"].cpu(), d["W"].cpu(), d["targets"].cpu().numpy(),
                                        rows, sup, tau, dtype)
    _abs(logp, o["logp"], "logp (support 2^-%d)" % j)
    _abs(ent, o["ent"], "ent (support 2^-%d)" % j)


@pytest.mark.parametrize("case", CASES[2::3], ids=[_id(c) for c in CASES[2::3]])
def test_support_backward_sweep(case):
    T, H, V, dtype, tau, rows, seed = case
    d = _scaled("bwd", T, H, V, dtype, tau, seed)
    j = int(_extra(case, 3).integers(0, 4))
    sup = workloads.support_words(T, V, j, seed % (2**31), targets=d["targets"].cpu().numpy())
    n = T if rows is None else len(rows)
    g = np.random.Generator(np.random.PCG64([seed, 8]))
    g1 = torch.from_numpy(g.standard_normal(n, dtype=np.float32)).cuda()
    g2 = torch.from_numpy(g.standard_normal(n, dtype=np.float32)).cuda()
    ri = None if rows is None else torch.from_numpy(rows).cuda()
    dh, dW = flp.backward(d["h"], d["W"], d["targets"], ri, tau, g1, g2,
                          support=torch.from_numpy(sup).cuda())
    torch.cuda.synchronize()
    dh_rows, ref_dW = coracle.backward_support(d["h"].cpu(), d["W"].cpu(),
                                               d["targets"].cpu().numpy(), rows, sup, tau,
                                               g1.cpu().numpy(), g2.cpu().numpy(), dtype)
    ref_dh = coracle.scatter_rows(dh_rows, np.arange(T) if rows is None else rows, T)
    _rel_or_zero(dh, ref_dh, "dh (support 2^-%d)" % j)
    _rel_or_zero(dW, ref_dW, "dW (support 2^-%d)" % j)


MX_CASES = [c for c in CASES if c[3] == "bf16"][::2]


@pytest.mark.parametrize("case", MX_CASES, ids=[_id(c) for c in MX_CASES])
def test_kl_mxfp4_sweep(case):
    """The teacher head quantised to MXFP4 (bf16 workloads: the decoded
    teacher weights meet bf16 hidden states in the MMA).  The MXFP4 layout
    takes whole 64-wide column blocks, so H is rounded up to a multiple of
    64."""
    T, H, V, _, _, rows, seed = case
    H = 64 * ((H + 63) // 64)
    d = _scaled("kl", T, H, V, "bf16", 1.0, seed)
    packed, scales = flp.mxfp4_quantize(d["W_t"])
    ri = None if rows is None else torch.from_numpy(rows).cuda()
    kl = flp.kl_divergence_mxfp4(d["h_s"], d["W_s"], d["h_t"], packed, scales, ri)
    torch.cuda.synchronize()
    opacked, oscales = coracle.mxfp4_quantize(d["W_t"].cpu(), "bf16")   # the oracle's own
    want = coracle.kl_mxfp4(d["h_s"].cpu(), d["W_s"].cpu(), d["h_t"].cpu(), opacked, oscales,
                            rows, "bf16")
    _abs(kl, want, "kl (MXFP4 teacher)")


BS_CASES = CASES[1::3]


@pytest.mark.parametrize("case", BS_CASES, ids=[_id(c) for c in BS_CASES])
def test_kl_block_scaled_sweep(case):
    """The teacher on the block-scaled tensor cores (MXFP8 rows, MXFP4 head),
    bf16 and fp16; the layout takes whole 128-wide k-chunks, so H is rounded
    up to a multiple of 128."""
    T, H, V, dtype, _, rows, seed = case
    H = 128 * ((H + 127) // 128)
    d = _scaled("kl", T, H, V, dtype, 1.0, seed)
    head = flp.mx_head_quantize(d["W_t"])
    ri = None if rows is None else torch.from_numpy(rows).cuda()
    kl = flp.kl_divergence_mx(d["h_s"], d["W_s"], d["h_t"], head, ri)
    torch.cuda.synchronize()
    packed, scales = coracle.mxfp4_quantize(d["W_t"].cpu(), dtype)
    want = coracle.kl_mx(d["h_s"].cpu(), d["W_s"].cpu(), d["h_t"].cpu(), packed, scales, rows,
                         dtype)
    _abs(kl, want, "kl (block-scaled teacher)")


MXF_CASES = CASES[2::3]


@pytest.mark.parametrize("case", MXF_CASES, ids=[_id(c) for c in MXF_CASES])
def test_forward_block_scaled_sweep(case):
    """Scoring on the block-scaled tensor cores (MXFP8 rows, MXFP4 head),
    bf16 and fp16, the case's temperature and rows; H rounded up to a
    multiple of 128 (whole k-chunks)."""
    T, H, V, dtype, tau, rows, seed = case
    H = 128 * ((H + 127) // 128)
    d = _scaled("fwd", T, H, V, dtype, tau, seed)
    head = flp.mx_head_quantize(d["W"])
    ri = None if rows is None else torch.from_numpy(rows).cuda()
    logp, ent, lse, ez = flp.logprob_entropy_mx(d["h"], head, V, d["targets"], ri, tau,
                                                return_stats=True)
    torch.cuda.synchronize()
    packed, scales = coracle.mxfp4_quantize(d["W"].cpu(), dtype)
    o = coracle.logprob_entropy_mx(d["h"].cpu(), packed, scales, V, d["targets"].cpu().numpy(),
                                   rows, tau, dtype)
    _abs(logp, o["logp"], "logp (block-scaled)")
    _abs(ent, o["ent"], "ent (block-scaled)")
    _abs(lse, o["lse"], "lse (block-scaled)")
