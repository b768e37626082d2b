"""GPU parity of the block-scaled teacher path (flp_kl_mx and its quantisers).

* flp_mxfp8_quantize against the oracle's MXFP8 quantiser, bit for bit (bf16
  and fp16 rows; all-zero, tiny and subnormal blocks; ties and values that
  saturate at 448).
* flp_mx_head_quantize against the oracle's MXFP4 quantiser, bit for bit:
  the oracle's blocked codes and scales, re-laid into the head layout that
  include/fusedlogp.h documents (codes [V, H/2], 512-byte scale atoms per
  224-row tile and 128-wide k-chunk).
* flp_kl_mx against the float64 oracle's KL with MXFP8 teacher rows and an
  MXFP4 teacher head (orc_kl_mx), |d KL| <= 1e-3, on shapes that span
  several row and vocabulary tiles with ragged tails, with and without
  row_idx, bf16 and fp16; and on sampled rows of the full distillation
  workload (8192 x 4096 x 129,280).  The oracle's quantised operands come
  from the oracle's own quantisers, never from the GPU.
* A student equal to the dequantised teacher (every MXFP8 and MXFP4 value is
  a bf16 value) gives KL = 0 up to FP32 rounding.
"""
import numpy as np
import pytest
import torch

import entropy_tcgen05_vocab_gb300 as flp
import workloads
from oracle import coracle, ref

pytestmark = pytest.mark.gpu
TOL = 1e-3
TILE = 224      # vocabulary rows per tile of the head's scale atoms


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    flp.build()
    flp.lib()


def _dt(x):
    return "bf16" if x.dtype == torch.bfloat16 else "fp16"


def _rows_with_edges(R, H, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    X = torch.randn(R, H, generator=g) * torch.exp(torch.randn(R, 1, generator=g) * 2)
    X[0, :32] = 0.0                                        # all-zero block
    X[1, 32:64] = 1e-30 if dtype == torch.bfloat16 else 1e-6   # tiny block
    # ties between E4M3 neighbours and values at / past the largest finite
    # value, in units of a block scale of 2^0 (max |x| in [256, 512))
    X[2, :16] = torch.tensor([256.0, 272.0, 288.0, 304.0, 320.0, 336.0, 352.0, 368.0,
                              384.0, 400.0, 416.0, 432.0, 448.0, 464.0, 480.0, 511.0])
    X[2, 16:32] = torch.tensor([0.0078125 * k for k in range(1, 17)])  # below the scale's grid
    X[3, :32] = -X[2, :32]
    if dtype == torch.bfloat16 and H >= 96:
        X[4, 64:96] = torch.linspace(-3e-39, 3e-39, 32)    # subnormal bf16 values
    # E4M3's subnormal steps (2^-9 at a block scale of 2^0), halfway cases
    # included: k 2^-10 lies halfway between two steps for every odd k
    X[5, 0] = 400.0
    X[5, 1:32] = torch.tensor([k * 2.0 ** -10 for k in range(1, 32)])
    return X.to(dtype)


@pytest.mark.parametrize("R,H,dtype", [(37, 128, torch.bfloat16), (300, 256, torch.float16),
                                       (129, 4096, torch.bfloat16), (64, 32, torch.bfloat16)])
def test_mxfp8_quantiser_matches_the_oracle_bit_for_bit(R, H, dtype):
    X = _rows_with_edges(R, H, dtype, seed=R + H)
    codes, scales = flp.mxfp8_quantize(X.cuda())
    oc, osc = coracle.mxfp8_quantize(X, _dt(X))
    assert np.array_equal(scales.cpu().numpy(), osc)
    got = codes.cpu().numpy()
    bad = np.argwhere(got != oc)
    assert bad.size == 0, (bad[:5], got[tuple(bad[0])], oc[tuple(bad[0])])


def test_mxfp8_quantiser_reads_a_strided_matrix():
    g = torch.Generator().manual_seed(3)
    big = torch.randn(100, 320, generator=g).to(torch.bfloat16).cuda()
    a = flp.mxfp8_quantize(big[:, :256])
    b = flp.mxfp8_quantize(big[:, :256].contiguous())
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def _head_from_oracle(packed, scales, V, H):
    """The head layout of include/fusedlogp.h, built from the oracle's blocked
    MXFP4 arrays ([H/64, V_pad, 32] codes, [H/64, V_pad, 2] scales)."""
    codes = packed[:, :V, :].transpose(1, 0, 2).reshape(V, H // 2)
    plain = scales[:, :V, :].transpose(1, 0, 2).reshape(V, H // 32)    # [V, H/32]
    kc_n = H // 128
    tiles = -(-V // TILE)
    atoms = np.zeros(tiles * kc_n * 1024, np.uint8)
    v = np.arange(V)[:, None]
    j = np.arange(H // 32)[None, :]
    t, i = v // TILE, v % TILE
    a, r = i // 128, i % 128
    off = ((t * kc_n + j // 4) * 2 + a) * 512 + (r % 32) * 16 + (r // 32) * 4 + j % 4
    atoms[off.ravel()] = plain.ravel()
    code_bytes = -(-V * H // 2 // 1024) * 1024
    out = np.zeros(code_bytes + atoms.size, np.uint8)
    out[:V * H // 2] = codes.ravel()
    out[code_bytes:] = atoms
    return out


@pytest.mark.parametrize("V,H,dtype", [(300, 128, torch.bfloat16), (1000, 256, torch.float16),
                                       (224, 512, torch.bfloat16), (4097, 384, torch.bfloat16)])
def test_head_quantiser_matches_the_oracle_bit_for_bit(V, H, dtype):
    g = torch.Generator().manual_seed(V * 7 + H)
    W = torch.randn(V, H, generator=g) * torch.exp(torch.randn(V, 1, generator=g) * 2)
    W[0, :32] = 0.0
    W[2, :8] = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.9])
    W = W.to(dtype)
    head = flp.mx_head_quantize(W.cuda())
    pc, sc = coracle.mxfp4_quantize(W, _dt(W))
    want = _head_from_oracle(pc, sc, V, H)
    assert head.numel() == want.size
    assert np.array_equal(head.cpu().numpy(), want)


def _case(T, H, V, seed, rows=False, dtype="bf16"):
    w = workloads.WORKLOADS[3].scaled(T=T, H=H, V=V, seed=seed, dtype=dtype)
    d = workloads.make(w, device="cuda")
    d["rows"] = None
    if rows:
        d["rows"] = torch.from_numpy(workloads.sample_rows(T, T // 2, seed=seed)).cuda()
    d["head"] = flp.mx_head_quantize(d["W_t"])
    d["dt"] = dtype
    return d


def _oracle_kl(d, rows):
    packed, scales = coracle.mxfp4_quantize(d["W_t"].cpu(), d["dt"])
    return coracle.kl_mx(d["h_s"].cpu(), d["W_s"].cpu(), d["h_t"].cpu(), packed, scales, rows,
                         d["dt"])


@pytest.mark.parametrize("T,H,V,rows,dtype", [
    (300, 256, 3000, False, "bf16"),     # two row tiles, 14 vocabulary tiles, ragged tails
    (129, 128, 300, True, "bf16"),       # one k-chunk; a tile of 76 columns
    (260, 512, 8200, True, "bf16"),
    (1000, 128, 20000, False, "bf16"),   # many tiles and splits
    (200, 384, 5000, False, "fp16"),
    (77, 1024, 224, False, "bf16"),      # exactly one vocabulary tile
])
def test_kl_mx_matches_the_oracle(T, H, V, rows, dtype):
    d = _case(T, H, V, seed=T + V + H, rows=rows, dtype=dtype)
    kl = flp.kl_divergence_mx(d["h_s"], d["W_s"], d["h_t"], d["head"], d["rows"])
    torch.cuda.synchronize()
    r = None if d["rows"] is None else d["rows"].cpu().numpy()
    want = _oracle_kl(d, r)
    got = kl.cpu().double().numpy()
    assert np.all(np.isfinite(got))
    err = np.abs(got - want).max()
    assert err <= TOL, err


def test_kl_mx_is_zero_against_the_dequantised_teacher():
    """Student = the teacher's quantised operands in bf16 (exact: E4M3 and
    E2M1 values times powers of two in range are bf16 values), so the two
    logit rows agree up to FP32 summation order and KL ~ 0."""
    T, H, V = 256, 512, 5000
    d = _case(T, H, V, seed=17)
    oc, osc = coracle.mxfp8_quantize(d["h_t"].cpu(), "bf16")
    hq = torch.from_numpy(ref.mxfp8_dequantize(oc, osc))
    pc, sc = coracle.mxfp4_quantize(d["W_t"].cpu(), "bf16")
    wq = torch.from_numpy(ref.mxfp4_dequantize(pc, sc, V))
    h_s, W_s = hq.to(torch.bfloat16), wq.to(torch.bfloat16)
    assert torch.equal(h_s.double(), hq) and torch.equal(W_s.double(), wq)
    kl = flp.kl_divergence_mx(h_s.cuda(), W_s.cuda(), d["h_t"], d["head"])
    assert kl.abs().max().item() <= 2e-5


def test_kl_mx_no_rows_and_argument_checks():
    d = _case(64, 128, 1000, seed=9)
    empty = torch.zeros(0, dtype=torch.int64, device="cuda")
    assert flp.kl_divergence_mx(d["h_s"], d["W_s"], d["h_t"], d["head"], empty).numel() == 0
    w = workloads.make(workloads.WORKLOADS[3].scaled(T=64, H=192, V=1000, seed=2), device="cuda")
    with pytest.raises(TypeError):               # H not a multiple of 128
        flp.mx_head_quantize(w["W_t"])
    shape = flp.make_shape(64, 192, 1000, 64, torch.bfloat16)
    assert flp.workspace_size(shape, flp.OP_KL_MX) == 0


def test_kl_mx_bad_row_index_is_counted():
    d = _case(200, 256, 3000, seed=21)
    rows = torch.tensor([0, 5, 199, 200, -1, 7], dtype=torch.int64, device="cuda")
    shape = flp.make_shape(200, 256, 3000, 6, torch.bfloat16)
    ws = torch.empty(flp.workspace_size(shape, flp.OP_KL_MX), dtype=torch.uint8, device="cuda")
    kl = flp.kl_divergence_mx(d["h_s"], d["W_s"], d["h_t"], d["head"], rows, workspace=ws)
    st = flp.read_device_status(ws)
    assert st["bad_rows"] == 2 and st["timeouts"] == 0
    got = kl.cpu().double().numpy()
    assert np.isnan(got[3]) and np.isnan(got[4])
    want = _oracle_kl(d, np.array([0, 5, 199, 7]))
    assert np.abs(got[[0, 1, 2, 5]] - want).max() <= TOL


def test_kl_mx_repeated_calls_are_bitwise_identical():
    d = _case(300, 256, 3000, seed=82)
    a = flp.kl_divergence_mx(d["h_s"], d["W_s"], d["h_t"], d["head"])
    b = flp.kl_divergence_mx(d["h_s"], d["W_s"], d["h_t"], d["head"])
    assert torch.equal(a, b)


def test_distill_workload_with_block_scaled_teacher_sampled():
    d = workloads.make(3, device="cuda")
    head = flp.mx_head_quantize(d["W_t"])
    kl = flp.kl_divergence_mx(d["h_s"], d["W_s"], d["h_t"], head)
    torch.cuda.synchronize()
    pos = np.unique(np.concatenate([workloads.sample_rows(8192, 48, seed=75), [0, 8191]]))
    packed, scales = coracle.mxfp4_quantize(d["W_t"].cpu(), "bf16")
    want = coracle.kl_mx(d["h_s"].cpu(), d["W_s"].cpu(), d["h_t"].cpu(), packed, scales, pos,
                         "bf16")
    got = kl[torch.from_numpy(pos).cuda()].cpu().double().numpy()
    assert np.abs(got - want).max() <= TOL
    allkl = kl.cpu().numpy()
    assert np.all(np.isfinite(allkl)) and np.all(allkl >= -1e-4)
