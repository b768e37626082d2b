"""The C ABI on the host (CPU only, no GPU calls).

Checks that libfusedlogp builds, loads and exports every function that
include/fusedlogp.h declares; that invalid arguments are rejected on the host
before anything is enqueued; the workspace formula; the tiling planner's
invariants; and the backward's row-chunk rule against the pages' printed
example and torch.chunk.
"""
import ctypes
import math
import os
import re

import pytest
import torch

import entropy_tcgen05_vocab_gb300 as flp
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = ctypes.c_void_p(1 << 20)   # never dereferenced: validation fails first


@pytest.fixture(scope="module")
def L():
    flp.build()
    return flp.lib()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(flp_\w+)\s*\(", src)
    return sorted(set(names))


def test_exports_every_declared_function(L):
    names = declared_functions()
    assert len(names) >= 9
    for nm in names:
        assert hasattr(L, nm), nm


def test_status_strings(L):
    for code in range(6):
        assert L.flp_status_string(code)
    assert L.flp_status_string(99) == b"unknown status"


def _shape(T=256, H=512, V=8192, n=256, dtype=0, ld_h=None, ld_w=None):
    return flp.FlpShape(T, H, V, n, dtype, H if ld_h is None else ld_h, H if ld_w is None else ld_w)


def _fwd(L, shape, tau=1.0, ws_bytes=1 << 40, ws=FAKE, h=FAKE, W=FAKE, row_idx=None,
         targets=FAKE, out=FAKE):
    return L.flp_logprob_entropy(ctypes.byref(shape) if shape is not None else None, h, W,
                                 targets, row_idx, tau, out, out, None, None, ws, ws_bytes, None)


@pytest.mark.parametrize("bad", [
    dict(H=0), dict(V=0), dict(T=-1), dict(n=-1), dict(H=100), dict(ld_h=500),
    dict(ld_w=516 + 2), dict(dtype=7)])
def test_invalid_shapes_rejected(L, bad):
    kw = dict(T=256, H=512, V=8192, n=256)
    kw.update(bad)
    assert _fwd(L, _shape(**kw)) == 1
    assert L.flp_last_error()
    assert L.flp_workspace_size(ctypes.byref(_shape(**kw)), 0) == 0


@pytest.mark.parametrize("tau", [0.0, -1.0, float("nan"), float("inf")])
def test_bad_temperature_rejected(L, tau):
    assert _fwd(L, _shape(), tau=tau) == 1
    assert b"temperature" in L.flp_last_error()


def test_host_validation_order(L):
    assert _fwd(L, None) == 1
    assert _fwd(L, _shape(), ws=None) == 3
    assert _fwd(L, _shape(), ws_bytes=100) == 3
    assert _fwd(L, _shape(), ws=ctypes.c_void_p((1 << 20) + 8)) == 1       # workspace alignment
    assert _fwd(L, _shape(n=200)) == 1                                     # row_idx NULL, n != T
    assert _fwd(L, _shape(), h=None) == 1
    assert _fwd(L, _shape(), h=ctypes.c_void_p((1 << 20) + 8)) == 1        # 16-byte alignment
    assert _fwd(L, _shape(), targets=None) == 1
    # nothing to score: valid and a no-op, even with null data pointers
    assert _fwd(L, _shape(n=0), row_idx=FAKE, h=None, W=None, targets=None, out=None) == 0


def test_kl_and_backward_validate_on_host(L):
    s = _shape()
    assert L.flp_kl(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, None, FAKE, None, 0, None) == 3
    assert L.flp_backward(ctypes.byref(s), FAKE, FAKE, FAKE, None, ctypes.c_float(1.0), FAKE,
                          FAKE, None, None, FAKE, FAKE, None, 0, None) == 3
    bad = _shape(H=12)
    assert L.flp_kl(ctypes.byref(bad), FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 1 << 40,
                    None) == 1
    # dh and dW may each be NULL (that gradient skipped), not both
    ws = 1 << 40
    assert L.flp_backward(ctypes.byref(s), FAKE, FAKE, FAKE, None, ctypes.c_float(1.0), FAKE,
                          FAKE, None, None, None, None, FAKE, ws, None) == 1
    assert b"both NULL" in L.flp_last_error()


def test_workspace_formula(L):
    for wid, w in workloads.WORKLOADS.items():
        n = {"all": w.T, "packed": 29492, "bernoulli": 9843}[w.rows]
        s = _shape(T=w.T, H=w.H, V=w.V, n=n)
        for op in (0, 1, 2):
            b = L.flp_workspace_size(ctypes.byref(s), op)
            assert b > 0
            gathered = n * w.H * 2 * (2 if op == 1 else 1)
            assert b >= gathered
            if op in (0, 1):
                # per-row state only (at most 64 splits x 2 column halves x 5
                # floats): far below a [n, V] FP32 logit buffer
                assert b - gathered <= n * 128 * 4 * 5 + (1 << 20)
                if w.V >= 38016:
                    assert b < n * w.V * 4
            else:
                assert b <= gathered + n * 128 * 4 * 4 + (4 << 30) + 4 * w.T + (1 << 20)
    # the block-scaled KL: gathered student rows, the teacher rows in MXFP8
    # (n*H bytes) and their scale atoms (n*H/32 bytes, whole 128-row blocks),
    # plus the same per-row state; 0 when H is not a multiple of 128
    w = workloads.WORKLOADS[3]
    s = _shape(T=w.T, H=w.H, V=w.V, n=w.T)
    b = L.flp_workspace_size(ctypes.byref(s), 3)
    q8 = w.T * w.H + (w.T + 127) // 128 * (w.H // 128) * 512
    assert q8 + w.T * w.H * 2 <= b <= q8 + w.T * w.H * 2 + w.T * 128 * 4 * 5 + (1 << 20)
    assert L.flp_workspace_size(ctypes.byref(_shape(T=64, H=192, V=1000, n=64)), 3) == 0
    # the block-scaled forward: the scored rows in MXFP8 and their atoms (no
    # gathered bf16 rows: the quantiser gathers), plus the forward's per-row
    # state and target logits
    w = workloads.WORKLOADS[1]
    s = _shape(T=w.T, H=w.H, V=w.V, n=w.T)
    b = L.flp_workspace_size(ctypes.byref(s), 4)
    q8 = w.T * w.H + (w.T + 127) // 128 * (w.H // 128) * 512
    assert q8 <= b <= q8 + w.T * 128 * 4 * 5 + (1 << 20)
    assert b < L.flp_workspace_size(ctypes.byref(s), 0)
    assert L.flp_workspace_size(ctypes.byref(_shape(T=64, H=192, V=1000, n=64)), 4) == 0
    assert L.flp_workspace_size(ctypes.byref(s), 5) == 0
    # monotone in the number of scored rows
    a = L.flp_workspace_size(ctypes.byref(_shape(T=4096, H=4096, V=151936, n=1000)), 0)
    b = L.flp_workspace_size(ctypes.byref(_shape(T=4096, H=4096, V=151936, n=2000)), 0)
    assert b > a


def test_mx_head_layout_sizes(L):
    """flp_mx_head_bytes: the E2M1 codes (V*H/2, rounded up to 1 KiB) and two
    512-byte scale atoms per 224-row vocabulary tile and 128-wide k-chunk."""
    L.flp_mx_head_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    L.flp_mx_head_bytes.restype = ctypes.c_size_t
    for V, H in ((129280, 4096), (224, 128), (225, 256), (1, 128)):
        codes = -(-V * H // 2 // 1024) * 1024
        assert L.flp_mx_head_bytes(V, H) == codes + -(-V // 224) * (H // 128) * 1024
    assert L.flp_mx_head_bytes(1000, 192) == 0 and L.flp_mx_head_bytes(0, 128) == 0
    # the workload-3 teacher head: 4 bits per weight plus a scale byte per 32
    # weights, in atoms of 256 row slots per 224-row tile
    bits = 8 * L.flp_mx_head_bytes(129280, 4096) / (129280 * 4096)
    assert abs(bits - (4 + 8 / 32 * 256 / 224)) < 1e-3


@pytest.mark.parametrize("wid", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("sms", [152, 148, 7])
def test_planner_covers_all_tiles_and_balances(L, wid, sms):
    w = workloads.WORKLOADS[wid]
    n = {"all": w.T, "packed": 29492, "bernoulli": 9843}[w.rows]
    op = 1 if w.kind == "kl" else 0
    p = flp.plan(_shape(T=w.T, H=w.H, V=w.V, n=n), op, sms)
    bn = 256 if op == 1 else 512
    cg = p["cta_group"]
    assert cg in (1, 2) and p["block_m"] == 128 * cg
    assert p["block_n"] == bn
    assert p["row_tiles"] == math.ceil(n / p["block_m"])
    assert p["vocab_tiles"] == math.ceil(w.V / bn)
    assert 1 <= p["splits"] <= 64
    S, tps = p["splits"], p["tiles_per_split"]
    assert tps * (S - 1) < p["vocab_tiles"] <= tps * S       # every split non-empty
    assert p["items"] == p["row_tiles"] * S
    units = max(1, sms // cg)
    assert p["grid"] == cg * min(p["items"], units)
    total = p["row_tiles"] * p["vocab_tiles"]
    ideal = math.ceil(total / (p["grid"] // cg))
    assert ideal <= p["max_tiles_per_cta"] <= ideal + tps
    if total >= 50 * units:
        assert p["max_tiles_per_cta"] <= 1.04 * total / units + 1


@pytest.mark.parametrize("n,V", [(4096, 151936), (256, 8192), (1, 224), (29492, 38016)])
def test_planner_block_scaled_ops(L, n, V):
    """The block-scaled KL plans 256 x 224 pair tiles and the block-scaled
    forward 256 x 448 (two head tiles), every split non-empty."""
    for op, bn in ((3, 224), (4, 448)):
        p = flp.plan(_shape(T=n, H=4096, V=V, n=n), op, 152)
        assert p["cta_group"] == 2 and p["block_m"] == 256 and p["block_n"] == bn
        assert p["vocab_tiles"] == math.ceil(V / bn)
        S, tps = p["splits"], p["tiles_per_split"]
        assert tps * (S - 1) < p["vocab_tiles"] <= tps * S
        assert p["items"] == p["row_tiles"] * S and p["grid"] == 2 * min(p["items"], 76)


def test_row_chunks_match_the_pages_example(L):
    rows = [list(map(int, ln.split())) for ln in open(os.path.join(ROOT, "tests", "golden",
                                                                     "chunk_shapes.txt"))
            if ln.strip() and not ln.startswith("#")]
    for n, c, *lengths in rows:
        assert flp.row_chunks(n, c) == lengths


@pytest.mark.parametrize("n,c", [(1, 1), (9, 4), (10, 4), (4096, 4096), (9843, 4096),
                                 (100, 7), (7, 100), (129, 128)])
def test_row_chunks_follow_torch_chunk(L, n, c):
    want = [t.numel() for t in torch.arange(n).chunk((n - 1) // c + 1)]
    assert flp.row_chunks(n, c) == want
    assert flp.row_chunks(0, c) == []


@pytest.mark.parametrize("limit", [0, 999_999, 2_000_000_000])
def test_selftest_limit_is_validated_on_host(L, limit):
    assert L.flp_selftest_wait_timeout(limit, FAKE, None) == 1
    assert L.flp_selftest_wait_timeout(50_000_000, None, None) == 3


@pytest.mark.parametrize("limit,ok", [(0, True), (99, False), (100, True), (60_000_000_000, True),
                                      (60_000_000_001, False)])
def test_wait_limit_is_validated_on_host(L, limit, ok):
    try:
        assert (L.flp_set_wait_limit(limit) == 0) == ok
    finally:
        assert L.flp_set_wait_limit(0) == 0


def test_scoring_without_row_idx_needs_no_room_for_gathered_rows(L):
    """The scoring and KL calls gather no rows when row_idx is NULL, so a
    workspace smaller by the gathered rows' bytes passes the workspace check
    (the call then fails later, on the device query, since there is no GPU
    here); with row_idx the same workspace is rejected as too small."""
    T, H, V = 4096, 4096, 151936
    s = _shape(T=T, H=H, V=V, n=T)
    for op, heads in ((0, 1), (1, 2)):
        full = L.flp_workspace_size(ctypes.byref(s), op)
        small = full - heads * T * H * 2
        if op == 0:
            assert _fwd(L, s, ws_bytes=small) != 3
            assert _fwd(L, s, ws_bytes=small, row_idx=FAKE) == 3
        else:
            kl = lambda ri: L.flp_kl(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, ri, FAKE, FAKE,
                                     small, None)
            assert kl(None) != 3
            assert kl(FAKE) == 3
        assert L.flp_workspace_size(ctypes.byref(s), op) == full


def test_noalloc_scratch_limit_on_host(L):
    """flp_logprob_entropy_noalloc's 16 MiB static scratch holds the forward
    of 4096 x 4096 x 151,936 without row_idx, and of up to 1,718 gathered
    rows at that H and V; more gathered rows are rejected before any device
    call."""
    lim = 16 << 20
    nofit = _shape(T=4096, H=4096, V=151936, n=1719)
    assert L.flp_workspace_size(ctypes.byref(nofit), 0) > lim
    fit = _shape(T=4096, H=4096, V=151936, n=1718)
    assert L.flp_workspace_size(ctypes.byref(fit), 0) <= lim
    call = lambda s, ri: L.flp_logprob_entropy_noalloc(ctypes.byref(s), FAKE, FAKE, FAKE, ri, 1.0,
                                                       FAKE, FAKE, None, None, None)
    assert call(nofit, FAKE) == 3
    assert b"static scratch" in L.flp_last_error()
    assert call(fit, FAKE) != 3                              # fails later: no GPU here
    assert call(_shape(T=4096, H=4096, V=151936, n=4096), None) != 3


def test_support_entry_points_validate_on_host(L):
    s = _shape()                       # V = 8192: 256 words per row
    sup = ctypes.c_void_p(1 << 21)

    def fwd(support=sup, ld=256, ws_bytes=1 << 40):
        return L.flp_logprob_entropy_support(ctypes.byref(s), FAKE, FAKE, FAKE, None, support, ld,
                                             ctypes.c_float(1.0), FAKE, FAKE, None, None, FAKE,
                                             ctypes.c_size_t(ws_bytes), None)

    assert fwd(support=None) == 1
    assert fwd(ld=255) == 1
    assert b"ld_support" in L.flp_last_error()
    assert fwd(support=ctypes.c_void_p((1 << 21) + 2)) == 1      # 4-byte alignment
    assert fwd(ws_bytes=10) == 3

    def bwd(support=sup, ld=256):
        return L.flp_backward_support(ctypes.byref(s), FAKE, FAKE, FAKE, None, support, ld,
                                      ctypes.c_float(0.7), FAKE, FAKE, None, None, FAKE, FAKE,
                                      FAKE, ctypes.c_size_t(1 << 40), None)

    assert bwd(support=None) == 1
    assert bwd(ld=100) == 1
    i64 = ctypes.c_int64
    pack = L.flp_pack_support
    assert pack(FAKE, i64(4), i64(70), i64(69), sup, i64(3), None) == 1       # ld_mask < V
    assert pack(FAKE, i64(4), i64(70), i64(70), sup, i64(2), None) == 1       # ld_support < 3
    assert pack(FAKE, i64(4), i64(0), i64(70), sup, i64(3), None) == 1        # V = 0
    assert pack(None, i64(0), i64(70), i64(70), None, i64(3), None) == 0      # nothing to pack
    assert pack(None, i64(4), i64(70), i64(70), sup, i64(3), None) == 1


def test_mxfp4_layout_sizes(L):
    assert L.flp_mxfp4_rows(1) == 256 and L.flp_mxfp4_rows(256) == 256
    assert L.flp_mxfp4_rows(257) == 512 and L.flp_mxfp4_rows(0) == 0
    assert L.flp_mxfp4_rows(129280) == 129280
    pb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    tot = L.flp_mxfp4_bytes(1000, 128, ctypes.byref(pb), ctypes.byref(sb))
    assert pb.value == 2 * 1024 * 32 and sb.value == 2 * 1024 * 2 and tot == pb.value + sb.value
    assert L.flp_mxfp4_bytes(1000, 100, None, None) == 0
    # 4.25 bits per weight plus the row padding, against 16 for bf16
    assert L.flp_mxfp4_bytes(129280, 4096, None, None) == 129280 * 4096 * 17 // 32


def test_mxfp4_entry_points_validate_on_host(L):
    s = _shape()
    assert L.flp_kl_mxfp4(ctypes.byref(s), FAKE, FAKE, FAKE, None, FAKE, None, FAKE, FAKE,
                          ctypes.c_size_t(1 << 40), None) == 1          # packed missing
    assert L.flp_kl_mxfp4(ctypes.byref(s), FAKE, FAKE, FAKE, ctypes.c_void_p((1 << 20) + 8), FAKE,
                          None, FAKE, FAKE, ctypes.c_size_t(1 << 40), None) == 1   # alignment
    half = _shape(dtype=1)
    assert L.flp_kl_mxfp4(ctypes.byref(half), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE,
                          ctypes.c_size_t(1 << 40), None) == 2          # fp16: unsupported
    odd = _shape(H=520, ld_h=520, ld_w=520)
    assert L.flp_kl_mxfp4(ctypes.byref(odd), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE,
                          ctypes.c_size_t(1 << 40), None) == 1          # H % 64
    i64 = ctypes.c_int64
    assert L.flp_mxfp4_quantize(FAKE, 0, i64(100), i64(96), i64(96), FAKE, FAKE, None) == 1
    assert L.flp_mxfp4_quantize(FAKE, 0, i64(100), i64(128), i64(64), FAKE, FAKE, None) == 1
    assert L.flp_mxfp4_quantize(None, 0, i64(100), i64(128), i64(128), FAKE, FAKE, None) == 1


def test_block_scaled_forward_validates_on_host(L):
    f = L.flp_logprob_entropy_mx
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_float] + [ctypes.c_void_p] * 5 + \
        [ctypes.c_size_t, ctypes.c_void_p]
    s = _shape(H=512, ld_h=512, ld_w=512)
    big = ctypes.c_size_t(1 << 40)
    ok = [FAKE, FAKE, FAKE, None, 0.7, FAKE, FAKE, None, None, FAKE, big, None]
    def call(shape, **kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(ctypes.byref(shape), *a)
    assert call(_shape(H=520, ld_h=520, ld_w=520)) == 1                  # H % 128
    assert call(s, a4=0.0) == 1 and call(s, a4=float("nan")) == 1        # temperature
    assert call(s, a1=None) == 1                                         # head missing
    assert call(s, a1=ctypes.c_void_p((1 << 20) + 16)) == 1              # head alignment
    assert call(s, a0=ctypes.c_void_p((1 << 20) + 8)) == 1               # h alignment
    assert call(s, a9=None) == 3                                         # workspace
    assert call(s, a10=ctypes.c_size_t(16)) == 3
    # a vocabulary whose scale atoms would pass the 32-bit coordinates of the
    # tiling (cdiv(V, 224) * H/128 * 64 rows of atoms); rejected on the host
    huge = _shape(T=256, H=4096, V=300_000_000, n=256, ld_h=4096, ld_w=4096)
    assert call(huge) == 1 and "tiling range" in flp.lib().flp_last_error().decode()
    assert L.flp_kl_mx(ctypes.byref(huge), FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, big,
                       None) == 1


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the built .so every entry point raises: there is no CPU or
    PyTorch fallback for the product path."""
    monkeypatch.setattr(flp._build, "LIB", str(tmp_path / "absent.so"))
    monkeypatch.setattr(flp, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        flp.lib()
    h = torch.zeros(4, 64, dtype=torch.bfloat16)
    with pytest.raises((RuntimeError, TypeError)):
        flp.logprob_entropy(h, h, torch.zeros(4, dtype=torch.int64))


def test_product_package_does_not_import_the_oracle():
    import ast
    pkg = os.path.join(ROOT, "entropy_tcgen05_vocab_gb300")
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            tree = ast.parse(open(os.path.join(pkg, fn)).read())
            for node in ast.walk(tree):
                mods = []
                if isinstance(node, ast.Import):
                    mods = [a.name for a in node.names]
                elif isinstance(node, ast.ImportFrom):
                    mods = [node.module or ""]
                assert not any(m == "oracle" or m.startswith("oracle.") for m in mods), fn


def test_plain_c_caller_compiles_against_the_header(L, tmp_path):
    """The public header is plain C: a C11 caller (tests/c_caller) compiles
    and links against the library with gcc -Wall -Werror.  Running it needs a
    GPU (tests/test_c_abi_gpu.py)."""
    import shutil
    import subprocess
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    if shutil.which("gcc") is None or not os.path.exists(os.path.join(cuda, "include", "cuda_runtime.h")):
        pytest.skip("gcc or the CUDA headers are missing")
    libdirs = [os.path.join(cuda, d) for d in ("lib64", "targets/sbsa-linux/lib",
                                                "targets/x86_64-linux/lib")]
    cudalib = next((p for p in libdirs if os.path.exists(os.path.join(p, "libcudart.so"))), None)
    if cudalib is None:
        pytest.skip("libcudart.so not found")
    libdir = os.path.dirname(flp._build.LIB)
    subprocess.run(["gcc", "-O2", "-std=c11", "-Wall", "-Werror",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    os.path.join(ROOT, "tests", "c_caller", "flp_c_caller.c"),
                    "-o", str(tmp_path / "caller"), "-L", libdir, "-lfusedlogp",
                    "-L", cudalib, "-lcudart"], check=True)


@pytest.mark.parametrize("sms,split,tail", [
    (152, 9, 8),     # 312 dh tiles on 76 pairs: 304 whole, the last 8 in 9 K segments
    (148, 4, 16),    # 74 pairs: 16 left over, at most 80 partial slots -> 4 segments
    (200, 6, 12),    # 100 pairs: 12 left over -> 6 segments (80 slots)
    (80, 1, 0),      # 40 pairs: a last wave of 32 is more than half full, no split
])
def test_dh_split_plan(L, monkeypatch, sms, split, tail):
    """The dh GEMM's last, partial wave (workload 4: 9,843 scored rows, one
    chunk, 39 x 8 output tiles of 256 x 512, K = V = 151,936) is split along
    K when it would leave at least half of the CTA pairs idle, into as many
    segments as idle pairs, partial-tile slots (80) and 16-k-block segments
    allow."""
    monkeypatch.delenv("FLP_DH_SPLIT", raising=False)
    p = flp.plan(_shape(T=16384, H=4096, V=151936, n=9843), 2, sms)
    assert p["chunk_rows"] == 9843
    assert (p["dh_split"], p["dh_tail_tiles"]) == (split, tail)
    assert tail * split <= 80 and tail * split <= sms // 2


def test_dh_split_off_and_short_vocabularies(L, monkeypatch):
    monkeypatch.delenv("FLP_DH_SPLIT", raising=False)
    # V <= 1984: fewer than 32 k-blocks of 64, i.e. than two 16-k-block
    # segments, so no split and no slots
    short = _shape(T=300, H=256, V=1984, n=300)
    assert flp.plan(short, 2, 152)["dh_split"] == 1
    longer = _shape(T=300, H=256, V=3000, n=300)
    assert flp.plan(longer, 2, 152)["dh_split"] == 2
    assert L.flp_workspace_size(ctypes.byref(longer), 2) > L.flp_workspace_size(ctypes.byref(short), 2)
    monkeypatch.setenv("FLP_DH_SPLIT", "0")
    assert flp.plan(longer, 2, 152)["dh_split"] == 1
    # the forward and the KL have no dh GEMM
    assert flp.plan(longer, 0, 152)["dh_split"] == 1
