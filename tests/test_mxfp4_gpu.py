"""GPU parity of the MXFP4 teacher head: flp_mxfp4_quantize bit for bit
against the oracle's quantiser, and flp_kl_mxfp4 against the float64 oracle
KL on the decoded teacher weights.

Cases span several row and vocabulary tiles with ragged tails (V not a
multiple of 256, so padded rows of the blocked layout are read), bf16 and
fp16 inputs to the quantiser, all-zero and tiny blocks; at the full
distillation size (8192 x 4096 x 129,280) KL is compared on sampled rows.
The GPU result is also compared with flp_kl on the decoded weights given as
a bf16 matrix (the same numbers through the bf16 path).  Tolerance:
|d KL| <= 1e-3.
"""
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


@pytest.mark.parametrize("V,H,dtype", [(300, 128, torch.bfloat16), (1000, 256, torch.float16),
                                       (256, 64, torch.bfloat16), (4097, 512, torch.bfloat16)])
def test_quantiser_matches_the_oracle_bit_for_bit(V, H, dtype):
    g = torch.Generator().manual_seed(V + H)
    W = torch.randn(V, H, generator=g) * torch.exp(torch.randn(V, 1, generator=g) * 2)
    W[0, :32] = 0.0                                  # all-zero block
    W[1, 32:64] = 1e-30 if dtype == torch.bfloat16 else 1e-6   # tiny block
    W[2, :8] = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.9])   # ties, saturation
    W = W.to(dtype)
    packed, scales = flp.mxfp4_quantize(W.cuda())
    pc, sc = coracle.mxfp4_quantize(W, _dt(W))
    assert np.array_equal(packed.cpu().numpy(), pc)
    assert np.array_equal(scales.cpu().numpy(), sc)


def test_quantiser_reads_a_strided_matrix():
    g = torch.Generator().manual_seed(5)
    big = torch.randn(500, 320, generator=g).to(torch.bfloat16).cuda()
    W = big[:, :256]
    assert W.stride(0) == 320
    a = flp.mxfp4_quantize(W)
    b = flp.mxfp4_quantize(W.contiguous())
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def _kl_case(T, H, V, seed, rows=False):
    w = workloads.WORKLOADS[3].scaled(T=T, H=H, V=V, seed=seed)
    d = workloads.make(w, device="cuda")
    d["rows"] = None
    if rows:
        d["rows"] = torch.from_numpy(workloads.sample_rows(T, T // 2, seed=seed)).cuda()
    d["packed"], d["scales"] = flp.mxfp4_quantize(d["W_t"])
    # the oracle's own quantisation of the teacher head (the oracle takes no
    # input from the GPU); the two agree bit for bit
    d["opacked"], d["oscales"] = coracle.mxfp4_quantize(d["W_t"].cpu(), "bf16")
    assert np.array_equal(d["packed"].cpu().numpy(), d["opacked"])
    assert np.array_equal(d["scales"].cpu().numpy(), d["oscales"])
    return d


@pytest.mark.parametrize("T,H,V,rows", [
    (300, 256, 3000, False),     # several row and vocabulary tiles, ragged tails
    (129, 64, 300, True),        # one 64-wide column block; padded rows read
    (260, 512, 8200, True),
    (1000, 128, 20000, False),   # many tiles and splits
])
def test_kl_mxfp4_matches_the_oracle(T, H, V, rows):
    d = _kl_case(T, H, V, seed=T + V, rows=rows)
    kl = flp.kl_divergence_mxfp4(d["h_s"], d["W_s"], d["h_t"], d["packed"], d["scales"], d["rows"])
    torch.cuda.synchronize()
    r = None if d["rows"] is None else d["rows"].cpu().numpy()
    want = coracle.kl_mxfp4(d["h_s"].cpu(), d["W_s"].cpu(), d["h_t"].cpu(),
                            d["opacked"], d["oscales"], r, "bf16")
    got = kl.cpu().double().numpy()
    assert np.all(np.isfinite(got))
    err = np.abs(got - want).max()
    assert err <= TOL, err
    # the same numbers through the bf16 KL path, with the decoded weights as bf16
    Wt_dec = torch.from_numpy(ref.mxfp4_dequantize(d["opacked"], d["oscales"], V))
    Wt_bf = Wt_dec.to(torch.bfloat16)
    assert torch.equal(Wt_bf.double(), Wt_dec)      # every decoded value is a bf16 value
    kl2 = flp.kl_divergence(d["h_s"], d["W_s"], d["h_t"], Wt_bf.cuda(), d["rows"])
    assert torch.allclose(kl, kl2, rtol=0, atol=2e-5)


def test_kl_mxfp4_no_rows_and_argument_checks():
    d = _kl_case(64, 128, 1000, seed=9)
    empty = torch.zeros(0, dtype=torch.int64, device="cuda")
    assert flp.kl_divergence_mxfp4(d["h_s"], d["W_s"], d["h_t"], d["packed"], d["scales"],
                                   empty).numel() == 0
    with pytest.raises(flp.FlpError):
        flp.kl_divergence_mxfp4(d["h_s"].half(), d["W_s"].half(), d["h_t"].half(), d["packed"],
                                d["scales"])


def test_distill_workload_with_mxfp4_teacher_sampled():
    d = workloads.make(3, device="cuda")
    packed, scales = flp.mxfp4_quantize(d["W_t"])
    kl = flp.kl_divergence_mxfp4(d["h_s"], d["W_s"], d["h_t"], packed, scales)
    torch.cuda.synchronize()
    pos = np.unique(np.concatenate([workloads.sample_rows(8192, 48, seed=74), [0, 8191]]))
    opacked, oscales = coracle.mxfp4_quantize(d["W_t"].cpu(), "bf16")
    want = coracle.kl_mxfp4(d["h_s"].cpu(), d["W_s"].cpu(), d["h_t"].cpu(), opacked, oscales, pos,
                            "bf16")
    got = kl[torch.from_numpy(pos).cuda()].cpu().double().numpy()
    assert np.abs(got - want).max() <= TOL
    allkl = kl.cpu().numpy()
    assert np.all(np.isfinite(allkl)) and np.all(allkl >= -1e-4)


def test_kl_mxfp4_repeated_calls_are_bitwise_identical():
    d = _kl_case(300, 256, 3000, seed=82)
    a = flp.kl_divergence_mxfp4(d["h_s"], d["W_s"], d["h_t"], d["packed"], d["scales"])
    b = flp.kl_divergence_mxfp4(d["h_s"], d["W_s"], d["h_t"], d["packed"], d["scales"])
    assert torch.equal(a, b)
