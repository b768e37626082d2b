"""GPU parity of the block-scaled forward (flp_logprob_entropy_mx).

The scored rows are quantised to MXFP8 inside the call and the logits are
formed against the MXFP4 head (flp_mx_head_quantize) by block-scaled MMAs.
The oracle (orc_logprob_entropy_mx) takes the same two quantisations from its
own quantisers -- never from the GPU -- and scores in float64.

* logp, entropy, LSE and E[z'] within 1e-3 of the oracle (E[z'] 2e-3) on
  shapes that span several row and vocabulary tiles with ragged tails (an
  odd number of 224-row head tiles, so the last tile's second MMA reads rows
  past the head), with and without row_idx, bf16 and fp16, several
  temperatures, and on sampled rows of the full forward-scoring workload
  (4096 x 4096 x 151,936).
* The bf16 forward on the dequantised operands (every E4M3 and E2M1 value
  times a power of two in range is a bf16 value) gives the same numbers up
  to FP32 summation order.
* A zero head gives logp = -ln V and entropy = ln V; bad rows and targets
  give NaN and are counted; no rows is a no-op; repeated calls agree bit
  for bit.
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


def _dt(x):
    return "bf16" if x.dtype == torch.bfloat16 else "fp16"


def _case(T, H, V, seed, dtype="bf16", rows=False):
    w = workloads.WORKLOADS[1].scaled(T=T, H=H, V=V, seed=seed, dtype=dtype, targets="uniform")
    d = workloads.make(w, device="cuda")
    d["rows"] = None
    if rows:
        d["rows"] = torch.from_numpy(workloads.sample_rows(T, T // 2, seed=seed)).cuda()
    d["head"] = flp.mx_head_quantize(d["W"])
    return d


def _oracle(d, rows, tau):
    packed, scales = coracle.mxfp4_quantize(d["W"].cpu(), _dt(d["W"]))
    return coracle.logprob_entropy_mx(d["h"].cpu(), packed, scales, d["W"].shape[0],
                                      d["targets"].cpu().numpy(), rows, tau, _dt(d["h"]))


def _cmp(got, want, what, tol=TOL):
    g = got.detach().cpu().double().numpy()
    assert np.all(np.isfinite(g)), what
    err = np.abs(g - want).max()
    assert err <= tol, "%s: max |diff| %.3e" % (what, err)


@pytest.mark.parametrize("T,H,V,rows,dtype,tau", [
    (300, 256, 3000, False, "bf16", 0.7),    # two row tiles, 7 tiles of 448, ragged tails
    (129, 128, 300, True, "bf16", 1.0),      # one k-chunk; one tile, second head tile past V
    (260, 512, 8200, True, "bf16", 2.5),
    (1000, 128, 20000, False, "bf16", 0.7),  # many tiles and splits
    (200, 384, 5000, False, "fp16", 1.0),
    (77, 1024, 448, False, "bf16", 0.3),     # exactly one tile
    (513, 256, 224, True, "bf16", 1.0),      # one head tile: the second MMA reads only padding
])
def test_logprob_entropy_mx_matches_the_oracle(T, H, V, rows, dtype, tau):
    d = _case(T, H, V, seed=T + V + H, dtype=dtype, rows=rows)
    V = d["W"].shape[0]
    logp, ent, lse, ez = flp.logprob_entropy_mx(d["h"], d["head"], V, d["targets"], d["rows"], tau,
                                                return_stats=True)
    torch.cuda.synchronize()
    r = None if d["rows"] is None else d["rows"].cpu().numpy()
    o = _oracle(d, r, tau)
    _cmp(logp, o["logp"], "logp")
    _cmp(ent, o["ent"], "ent")
    _cmp(lse, o["lse"], "lse")
    _cmp(ez, o["ez"], "ez", 2e-3)


def test_logprob_entropy_mx_is_the_bf16_forward_on_the_dequantised_operands():
    T, H, V = 384, 512, 6000
    d = _case(T, H, V, seed=31)
    oc, osc = coracle.mxfp8_quantize(d["h"].cpu(), "bf16")
    hq = torch.from_numpy(ref.mxfp8_dequantize(oc, osc))
    pc, sc = coracle.mxfp4_quantize(d["W"].cpu(), "bf16")
    wq = torch.from_numpy(ref.mxfp4_dequantize(pc, sc, V))
    hb, wb = hq.to(torch.bfloat16), wq.to(torch.bfloat16)
    assert torch.equal(hb.double(), hq) and torch.equal(wb.double(), wq)
    a = flp.logprob_entropy(hb.cuda(), wb.cuda(), d["targets"], None, 0.7, return_stats=True)
    b = flp.logprob_entropy_mx(d["h"], d["head"], V, d["targets"], None, 0.7, return_stats=True)
    for x, y in zip(a, b):
        assert (x - y).abs().max().item() <= 2e-5


def test_logprob_entropy_mx_zero_head_closed_form():
    T, H, V = 260, 256, 5000
    d = _case(T, H, V, seed=41)
    head = flp.mx_head_quantize(torch.zeros(V, H, dtype=torch.bfloat16, device="cuda"))
    logp, ent = flp.logprob_entropy_mx(d["h"], head, V, d["targets"], None, 0.7)
    assert (logp + math.log(V)).abs().max().item() <= 1e-5
    assert (ent - math.log(V)).abs().max().item() <= 1e-5


def test_logprob_entropy_mx_bad_rows_and_targets():
    d = _case(200, 256, 3000, seed=23)
    tg = d["targets"].clone()
    tg[5] = 3000
    tg[7] = -2
    rows = torch.tensor([0, 5, 199, 200, -1, 7, 9], dtype=torch.int64, device="cuda")
    shape = flp.make_shape(200, 256, 3000, 7, torch.bfloat16)
    ws = torch.empty(flp.workspace_size(shape, flp.OP_LOGPROB_ENTROPY_MX), dtype=torch.uint8,
                     device="cuda")
    logp, ent = flp.logprob_entropy_mx(d["h"], d["head"], 3000, tg, rows, 1.0, workspace=ws)
    st = flp.read_device_status(ws)
    assert st["bad_rows"] == 2 and st["bad_targets"] == 2 and st["timeouts"] == 0
    lp, en = logp.cpu().double().numpy(), ent.cpu().double().numpy()
    assert np.all(np.isnan(lp[[1, 3, 4, 5]])) and np.all(np.isnan(en[[3, 4]]))
    ok = [0, 2, 6]
    o = _oracle(d, np.array([0, 199, 9]), 1.0)
    assert np.abs(lp[ok] - o["logp"]).max() <= TOL
    assert np.abs(en[[0, 1, 2, 5, 6]] - _oracle(d, np.array([0, 5, 199, 7, 9]), 1.0)["ent"]).max() \
        <= TOL


def test_logprob_entropy_mx_no_rows_and_argument_checks():
    d = _case(64, 128, 1000, seed=9)
    empty = torch.zeros(0, dtype=torch.int64, device="cuda")
    logp, ent = flp.logprob_entropy_mx(d["h"], d["head"], 1000, d["targets"], empty)
    assert logp.numel() == 0 and ent.numel() == 0
    shape = flp.make_shape(64, 192, 1000, 64, torch.bfloat16)
    assert flp.workspace_size(shape, flp.OP_LOGPROB_ENTROPY_MX) == 0   # H % 128 != 0
    with pytest.raises(TypeError):                                     # head too small
        flp.logprob_entropy_mx(d["h"], d["head"][:100], 1000, d["targets"])
    with pytest.raises(flp.FlpError):                                  # temperature
        flp.logprob_entropy_mx(d["h"], d["head"], 1000, d["targets"], None, 0.0)


def test_logprob_entropy_mx_repeated_calls_are_bitwise_identical():
    d = _case(300, 256, 3000, seed=83)
    a = flp.logprob_entropy_mx(d["h"], d["head"], 3000, d["targets"])
    b = flp.logprob_entropy_mx(d["h"], d["head"], 3000, d["targets"])
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_forward_scoring_workload_with_block_scaled_head_sampled():
    d = workloads.make(1, device="cuda")
    V = d["W"].shape[0]
    head = flp.mx_head_quantize(d["W"])
    logp, ent = flp.logprob_entropy_mx(d["h"], head, V, d["targets"], None, d["tau"])
    torch.cuda.synchronize()
    pos = np.unique(np.concatenate([workloads.sample_rows(4096, 40, seed=76), [0, 4095]]))
    packed, scales = coracle.mxfp4_quantize(d["W"].cpu(), "bf16")
    o = coracle.logprob_entropy_mx(d["h"].cpu(), packed, scales, V, d["targets"].cpu().numpy(),
                                   pos, d["tau"], "bf16")
    idx = torch.from_numpy(pos).cuda()
    _cmp(logp[idx], o["logp"], "logp")
    _cmp(ent[idx], o["ent"], "ent")
    lp, en = logp.cpu().numpy(), ent.cpu().numpy()
    assert np.all(np.isfinite(lp)) and np.all(lp <= 1e-4)
    assert np.all((en >= -1e-4) & (en <= math.log(V) + 1e-4))
