"""The C ABI from a plain C program: no Python binding and no torch in the
caller.  tests/c_caller/flp_c_caller.c is compiled with gcc against
include/fusedlogp.h and the built libfusedlogp.so, fed seeded inputs from
workloads.py through raw files, and its outputs (log-prob, entropy, KL with
a bf16 and with a block-scaled teacher, dh, dW) are compared with the float64 oracle: 1e-3 absolute for the per-row
values, 1e-2 relative (Frobenius) for the gradients.
"""
import os
import subprocess

import numpy as np
import pytest
import torch

import entropy_tcgen05_vocab_gb300 as flp
import workloads
from oracle import coracle

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_lib_dir(cuda):
    for d in ("lib64", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib", "lib"):
        p = os.path.join(cuda, d)
        if os.path.exists(os.path.join(p, "libcudart.so")):
            return p
    pytest.skip("libcudart.so not found under %s" % cuda)


def _bits(x):
    return x.detach().cpu().contiguous().view(torch.int16).numpy()


def test_plain_c_caller(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    flp.build()
    libdir = os.path.dirname(flp._build.LIB)
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cudalib = _cuda_lib_dir(cuda)
    exe = str(tmp_path / "flp_c_caller")
    subprocess.run(["gcc", "-O2", "-std=c11", "-Wall", "-Werror",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    os.path.join(ROOT, "tests", "c_caller", "flp_c_caller.c"), "-o", exe,
                    "-L", libdir, "-lfusedlogp", "-L", cudalib, "-lcudart",
                    "-Wl,-rpath," + libdir + ":" + cudalib], check=True)

    T, H, V = 300, 256, 5000
    d = workloads.make(workloads.WORKLOADS[4].scaled(T=T, H=H, V=V, seed=71), device="cpu")
    k = workloads.make(workloads.WORKLOADS[3].scaled(T=T, H=H, V=V, seed=72), device="cpu")
    rows = d["row_idx"].numpy()
    n = len(rows)
    for name, arr in (("h.bin", _bits(d["h"])), ("W.bin", _bits(d["W"])),
                      ("ht.bin", _bits(k["h_t"])), ("Wt.bin", _bits(k["W_t"])),
                      ("targets.bin", d["targets"].numpy().astype(np.int64)),
                      ("rows.bin", rows.astype(np.int64)),
                      ("g1.bin", d["g1"].numpy().astype(np.float32)),
                      ("g2.bin", d["g2"].numpy().astype(np.float32))):
        arr.tofile(str(tmp_path / name))
    r = subprocess.run([exe, str(tmp_path), str(T), str(H), str(V), str(n)],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr

    def out(name, dtype, shape):
        return np.fromfile(str(tmp_path / name), dtype=dtype).reshape(shape)

    tau = 0.7
    o = coracle.logprob_entropy(d["h"], d["W"], d["targets"].numpy(), rows, tau, "bf16")
    assert np.abs(out("logp.bin", np.float32, (n,)) - o["logp"]).max() <= 1e-3
    assert np.abs(out("ent.bin", np.float32, (n,)) - o["ent"]).max() <= 1e-3
    want_kl = coracle.kl(d["h"], d["W"], k["h_t"], k["W_t"], rows, "bf16")
    assert np.abs(out("kl.bin", np.float32, (n,)) - want_kl).max() <= 1e-3
    packed, scales = coracle.mxfp4_quantize(k["W_t"], "bf16")
    want_klmx = coracle.kl_mx(d["h"], d["W"], k["h_t"], packed, scales, rows, "bf16")
    assert np.abs(out("klmx.bin", np.float32, (n,)) - want_klmx).max() <= 1e-3
    # h scored against the teacher's head (MXFP4) on the block-scaled tensor cores
    omx = coracle.logprob_entropy_mx(d["h"], packed, scales, V, d["targets"].numpy(), rows, tau,
                                     "bf16")
    assert np.abs(out("logpmx.bin", np.float32, (n,)) - omx["logp"]).max() <= 1e-3
    assert np.abs(out("entmx.bin", np.float32, (n,)) - omx["ent"]).max() <= 1e-3
    dh_rows, dW = coracle.backward(d["h"], d["W"], d["targets"].numpy(), rows, tau,
                                   d["g1"].numpy(), d["g2"].numpy(), "bf16")
    dh = coracle.scatter_rows(dh_rows, rows, T)
    got_dh = torch.from_numpy(out("dh.bin", np.int16, (T, H))).view(torch.bfloat16).double().numpy()
    got_dW = out("dW.bin", np.float32, (V, H)).astype(np.float64)
    for got, want in ((got_dh, dh), (got_dW, dW)):
        assert np.linalg.norm(got - want) <= 1e-2 * np.linalg.norm(want)
