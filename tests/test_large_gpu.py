"""GPU parity past 2**31 elements.

h and W both have 1,048,700 rows of H = 2048 (2.15e9 elements, 4.3 GB each
in bf16), so the element offset of any row past 1,048,576 does not fit in 32
bits; the backward's dW (fp32, 8.6 GB) and dh have the same property.  The
scored rows are a seeded sample that includes the first and last rows of h
and the rows on either side of the 2**31 boundary; some targets are set to
vocabulary rows past it.  Each output is compared with the float64 C oracle
on those rows only (the oracle is given just the sampled rows of h):
log-prob and entropy within 1e-3, KL within 1e-3, dh and dW rows within the
backward tolerance (1e-2 of the reference's norm and of its largest entry).
The block-scaled forward scores every row of h, so its MXFP8 copy of the rows
in the workspace also passes 2**31 bytes.
"""
import numpy as np
import pytest
import torch

import entropy_tcgen05_vocab_gb300 as flp
import workloads
from oracle import coracle

pytestmark = pytest.mark.gpu
ROWS = 1_048_700          # rows of h and of W: ROWS * H > 2**31
H = 2048
EDGE = (1 << 31) // H     # first row whose element offset needs 33 bits


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    flp.build()
    flp.lib()


@pytest.fixture(scope="module")
def big():
    w = workloads.WORKLOADS[0].scaled(T=ROWS, H=H, V=ROWS, w_std=0.05, tau=0.7, seed=77)
    d = workloads.make(w, device="cuda")
    pos = np.unique(np.concatenate([workloads.sample_rows(ROWS, 20, seed=78),
                                    [0, EDGE - 1, EDGE, EDGE + 1, ROWS - 1]]))
    d["row_idx"] = torch.from_numpy(pos).cuda()
    # targets on either side of the boundary and at the last vocabulary row
    for i, t in zip(pos[-4:], (EDGE - 1, EDGE, ROWS - 2, ROWS - 1)):
        d["targets"][int(i)] = t
    d["pos"] = pos
    d["h_rows"] = d["h"][d["row_idx"]].cpu()
    d["W_cpu"] = d["W"].cpu()
    yield d
    d.clear()
    torch.cuda.empty_cache()


def _close(got, want, tol, what):
    g = got.detach().cpu().double().numpy()
    assert np.all(np.isfinite(g)), what + ": non-finite"
    err = np.abs(g - want).max()
    assert err <= tol, "%s: max |diff| %.3e" % (what, err)


def _rel(got, want, what, rtol=1e-2):
    g = got.detach().cpu().double().numpy()
    assert np.all(np.isfinite(g)), what + ": non-finite"
    fro = np.linalg.norm(g - want) / max(np.linalg.norm(want), 1e-30)
    ele = np.abs(g - want).max() / max(np.abs(want).max(), 1e-30)
    assert fro <= rtol and ele <= rtol, "%s: rel Frobenius %.2e, rel max %.2e" % (what, fro, ele)


def test_forward_past_32_bit_offsets(big):
    d = big
    logp, ent = flp.logprob_entropy(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"])
    torch.cuda.synchronize()
    tg = d["targets"][d["row_idx"]].cpu().numpy()
    o = coracle.logprob_entropy(d["h_rows"], d["W_cpu"], tg, None, d["tau"], "bf16")
    _close(logp, o["logp"], 1e-3, "logp")
    _close(ent, o["ent"], 1e-3, "ent")


def test_backward_past_32_bit_offsets(big):
    d = big
    n = d["row_idx"].shape[0]
    g1 = workloads.normal((n,), 1.0, 79, 1, "f32", "cpu").cuda()
    g2 = workloads.normal((n,), 1.0, 79, 2, "f32", "cpu").cuda()
    dh, dW = flp.backward(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"], g1, g2)
    torch.cuda.synchronize()
    tg = d["targets"][d["row_idx"]].cpu().numpy()
    vsel = np.array([0, 1, EDGE - 1, EDGE, EDGE + 1, ROWS - 2, ROWS - 1], np.int64)
    want_dh, want_dw = coracle.backward(d["h_rows"], d["W_cpu"], tg, None, d["tau"],
                                        g1.cpu().numpy(), g2.cpu().numpy(), "bf16", vsel=vsel)
    _rel(dh[d["row_idx"]], want_dh, "dh (scored rows)")
    _rel(dW[torch.from_numpy(vsel).cuda()], want_dw, "dW (rows across the boundary)")
    scored = torch.zeros(ROWS, dtype=torch.bool, device="cuda")
    scored[d["row_idx"]] = True
    assert torch.count_nonzero(dh[~scored]) == 0
    del dh, dW
    torch.cuda.empty_cache()


def test_kl_past_32_bit_offsets():
    w = workloads.WORKLOADS[3].scaled(T=24, H=H, V=ROWS, seed=80)
    d = workloads.make(w, device="cuda")
    kl = flp.kl_divergence(d["h_s"], d["W_s"], d["h_t"], d["W_t"])
    torch.cuda.synchronize()
    want = coracle.kl(d["h_s"].cpu(), d["W_s"].cpu(), d["h_t"].cpu(), d["W_t"].cpu(), None, "bf16")
    _close(kl, want, 1e-3, "kl")
    d.clear()
    torch.cuda.empty_cache()


def test_block_scaled_forward_past_32_bit_offsets(big):
    """Every row of h scored on the block-scaled tensor cores against a
    4096-row head: the MXFP8 rows in the workspace take 2.15e9 bytes, so
    their offsets, like h's, need 33 bits past row EDGE."""
    d = big
    Vs = 4096
    head = flp.mx_head_quantize(d["W"][:Vs].contiguous())
    tg = d["targets"] % Vs
    logp, ent = flp.logprob_entropy_mx(d["h"], head, Vs, tg, None, d["tau"])
    torch.cuda.synchronize()
    pos = d["pos"]
    packed, scales = coracle.mxfp4_quantize(d["W_cpu"][:Vs], "bf16")
    o = coracle.logprob_entropy_mx(d["h_rows"], packed, scales, Vs,
                                   tg[d["row_idx"]].cpu().numpy(), None, d["tau"], "bf16")
    idx = torch.from_numpy(pos).cuda()
    _close(logp[idx], o["logp"], 1e-3, "logp (block-scaled)")
    _close(ent[idx], o["ent"], 1e-3, "ent (block-scaled)")
    del head, logp, ent
    torch.cuda.empty_cache()
