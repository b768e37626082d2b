"""The no-allocation log-prob/entropy entry point, through the C ABI.

flp_logprob_entropy_noalloc serves callers that cannot give the library
device memory (no allocator of their own, a framework pool that has claimed
the device, or a loop where cudaMalloc's possible device synchronisation is
not allowed).  It keeps its scratch in one static device array inside the
library.  These tests call it directly through ctypes, twice in a row on
different problems, and compare each result with the workspace entry point
(flp_logprob_entropy) within the parity tolerance of the other GPU tests.
At the forward-scoring size (4096 rows, H 4096, V 151,936) without row_idx
the problem fits the 16 MiB array, and the result is checked against the
workspace entry point and the oracle.
This file is collected last so a failure here stops a run only after every
other test has run; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import entropy_tcgen05_vocab_gb300 as flp
import workloads

pytestmark = pytest.mark.gpu
TOL = 1e-3
SCRATCH_BYTES = 16 << 20          # FLP_NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    flp.build()
    return flp.lib()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(L, d, tau):
    h, W, ri = d["h"], d["W"], d["row_idx"]
    n = h.shape[0] if ri is None else ri.numel()
    shape = flp.make_shape(h.shape[0], h.shape[1], W.shape[0], n, h.dtype)
    logp = torch.empty(n, dtype=torch.float32, device="cuda")
    ent = torch.empty(n, dtype=torch.float32, device="cuda")
    lse = torch.empty(n, dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.flp_logprob_entropy_noalloc(ctypes.byref(shape), _ptr(h), _ptr(W), _ptr(d["targets"]),
                                       _ptr(ri), float(tau), _ptr(logp), _ptr(ent), _ptr(lse),
                                       None, stream)
    assert rc == 0, L.flp_last_error().decode()
    return logp, ent, lse


def _compare(got, want):
    g = got.cpu().double().numpy()
    w = want.cpu().double().numpy()
    assert np.all(np.isfinite(g))
    assert np.max(np.abs(g - w)) <= TOL


def test_noalloc_matches_workspace_entry_point_on_two_calls(L):
    # call 1: 256 x 512 x 8192 bf16, every row scored
    d1 = workloads.make(0, device="cuda")
    # call 2: packed fp16 rows selected by row_idx, another temperature
    d2 = workloads.make(workloads.WORKLOADS[2].scaled(T=2000, H=256, V=5000), device="cuda")
    for d, tau in ((d1, 1.0), (d2, 0.7)):
        logp, ent, lse = _noalloc(L, d, tau)
        ref_logp, ref_ent, ref_lse, _ = flp.logprob_entropy(d["h"], d["W"], d["targets"],
                                                            d["row_idx"], tau, return_stats=True)
        torch.cuda.synchronize()
        _compare(logp, ref_logp)
        _compare(ent, ref_ent)
        _compare(lse, ref_lse)


def test_noalloc_forward_scoring_size_without_row_idx(L):
    """4096 x 4096 x 151,936 bf16 at temperature 0.7 needs 6.1 MiB of scratch
    without row_idx: bitwise the workspace entry point's result (same
    kernels, same plan), and within 1e-3 of the float64 oracle on sampled
    rows."""
    from oracle import coracle
    d = workloads.make(1, device="cuda")
    assert d["row_idx"] is None
    logp, ent, lse = _noalloc(L, d, d["tau"])
    ref_logp, ref_ent, ref_lse, _ = flp.logprob_entropy(d["h"], d["W"], d["targets"], None,
                                                        d["tau"], return_stats=True)
    torch.cuda.synchronize()
    assert torch.equal(logp, ref_logp) and torch.equal(ent, ref_ent) and torch.equal(lse, ref_lse)
    sel = workloads.sample_rows(d["n"], 48, seed=11)
    o = coracle.logprob_entropy(d["h"].cpu(), d["W"].cpu(), d["targets"].cpu(), sel, d["tau"],
                                "bf16")
    assert np.abs(logp.cpu().double().numpy()[sel] - o["logp"]).max() <= TOL
    assert np.abs(ent.cpu().double().numpy()[sel] - o["ent"]).max() <= TOL


def test_noalloc_allocates_no_device_memory(L):
    """Neither torch's allocator nor the device's free memory changes over a
    call.  The free-memory check assumes no other process allocates on this
    GPU meanwhile.  The first call in a process may make CUDA load the
    library's module, which places the 16 MiB array (by design, once); so the
    free-memory comparison is taken on a later call, while torch's allocator
    is also checked across the first call of this test."""
    d = workloads.make(0, device="cuda")
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    _noalloc(L, d, 1.0)                  # first call on the device: address look-up
    torch.cuda.synchronize()
    # only the three [n] outputs _noalloc allocates itself (3 x 1 KiB blocks)
    assert torch.cuda.memory_allocated() - alloc0 <= 3 * 1024
    n = d["h"].shape[0]
    shape = flp.make_shape(n, 512, 8192, n, torch.bfloat16)
    outs = [torch.empty(n, dtype=torch.float32, device="cuda") for _ in range(2)]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc1 = torch.cuda.memory_allocated()
    rc = L.flp_logprob_entropy_noalloc(ctypes.byref(shape), _ptr(d["h"]), _ptr(d["W"]),
                                       _ptr(d["targets"]), None, 1.0, _ptr(outs[0]),
                                       _ptr(outs[1]), None, None, stream)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert rc == 0
    assert free1 == free0
    assert torch.cuda.memory_allocated() == alloc1


def test_noalloc_rejects_problems_beyond_the_static_scratch(L):
    # 4096 rows x H 4096 gathered through row_idx: the gathered rows alone
    # need 32 MiB > 16 MiB (without row_idx the same shape fits, above)
    shape = flp.make_shape(4096, 4096, 151936, 4096, torch.bfloat16)
    assert flp.workspace_size(shape, flp.OP_LOGPROB_ENTROPY) > SCRATCH_BYTES
    dummy = ctypes.c_void_p(1 << 20)
    rc = L.flp_logprob_entropy_noalloc(ctypes.byref(shape), dummy, dummy, dummy, dummy, 1.0,
                                       dummy, dummy, None, None, None)
    assert rc == 3
    assert b"static scratch" in L.flp_last_error()
